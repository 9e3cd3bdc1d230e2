// Offline MaskSpec compiler (host C++).
//
// Follows CompileMask section 3.2 (MaskSpec: query rows grouped into Regions, each with a row
// guard and a visibility rule) and section 3.2.2 (symbolic lowering of a visibility rule by AST
// construction, DNF normalisation, interval extraction and canonicalisation; the interval count
// is derived from the rules rather than fixed in advance).
//
//  parse      one Region per line: `region <guard> : <rule>`; AST of integer and boolean terms
//  DNF        negations pushed onto comparisons, `!=` split into `<` or `>`, AND distributed over
//             OR; each conjunct becomes one interval slot
//  extract    each comparison is solved for the other index j (coefficient +-1); lower bounds
//             combine with max, upper bounds with min; comparisons without j become the slot's
//             condition
//  canonical  integer terms are kept in a linear normal form (sum of coefficient x atom plus a
//             constant) so that equal endpoints compare equal; provably empty conjuncts and
//             constant conditions are folded, duplicate bounds and duplicate slots removed.
//             Two different slots are never merged: a merge must hold for every row of the
//             Region, which the symbolic form cannot show for the rules used here (e.g. the
//             Region C rule keeps [0, b) and [s(i), i + 1) as two slots).
//  emit       stack programs (program.h) evaluated per row by the generic preprocess kernel,
//             and the same endpoints as CUDA C++: the row evaluator of the spec's own
//             preprocess kernel, compiled at run time with NVRTC (codegen.cpp)
#include <algorithm>
#include <cctype>
#include <climits>
#include <cstdio>
#include <cstring>
#include <list>
#include <map>
#include <memory>
#include <atomic>
#include <mutex>
#include <sstream>
#include <stdexcept>
#include <string>
#include <vector>

#include "../../include/cm.h"
#include "program.h"

namespace cm {
namespace {

struct CompileError : std::runtime_error {
  using std::runtime_error::runtime_error;
};

// ---------------------------------------------------------------------------------------------
// lexer
// ---------------------------------------------------------------------------------------------
enum class T { Ident, Int, LParen, RParen, Comma, Plus, Minus, Star, Percent, Lt, Le, Gt, Ge, Eq,
               Ne, And, Or, Not, Colon, End };

struct Tok {
  T t;
  std::string s;
  long long v = 0;
  int col = 0;
};

std::vector<Tok> lex(const std::string& line, int lineno) {
  std::vector<Tok> out;
  size_t p = 0;
  auto err = [&](const std::string& m) {
    throw CompileError("line " + std::to_string(lineno) + ", col " + std::to_string(p + 1) +
                       ": " + m);
  };
  while (p < line.size()) {
    const char c = line[p];
    if (std::isspace(static_cast<unsigned char>(c))) { ++p; continue; }
    Tok k;
    k.col = static_cast<int>(p) + 1;
    if (std::isalpha(static_cast<unsigned char>(c)) || c == '_') {
      size_t q = p;
      while (q < line.size() && (std::isalnum(static_cast<unsigned char>(line[q])) || line[q] == '_')) ++q;
      k.t = T::Ident;
      k.s = line.substr(p, q - p);
      p = q;
    } else if (std::isdigit(static_cast<unsigned char>(c))) {
      size_t q = p;
      while (q < line.size() && std::isdigit(static_cast<unsigned char>(line[q]))) ++q;
      k.t = T::Int;
      k.s = line.substr(p, q - p);
      if (k.s.size() > 9) err("integer constant too large");
      k.v = std::stoll(k.s);
      p = q;
    } else {
      auto two = line.substr(p, 2);
      if (two == "<=") { k.t = T::Le; p += 2; }
      else if (two == ">=") { k.t = T::Ge; p += 2; }
      else if (two == "==") { k.t = T::Eq; p += 2; }
      else if (two == "!=") { k.t = T::Ne; p += 2; }
      else if (two == "&&") { k.t = T::And; p += 2; }
      else if (two == "||") { k.t = T::Or; p += 2; }
      else {
        switch (c) {
          case '(': k.t = T::LParen; break;
          case ')': k.t = T::RParen; break;
          case ',': k.t = T::Comma; break;
          case '+': k.t = T::Plus; break;
          case '-': k.t = T::Minus; break;
          case '*': k.t = T::Star; break;
          case '%': k.t = T::Percent; break;
          case '<': k.t = T::Lt; break;
          case '>': k.t = T::Gt; break;
          case '!': k.t = T::Not; break;
          case ':': k.t = T::Colon; break;
          default: err(std::string("unexpected character '") + c + "'");
        }
        ++p;
      }
    }
    out.push_back(k);
  }
  Tok e;
  e.t = T::End;
  e.col = static_cast<int>(line.size()) + 1;
  out.push_back(e);
  return out;
}

// ---------------------------------------------------------------------------------------------
// AST
// ---------------------------------------------------------------------------------------------
enum class EK { Const, I, J, S, Nseg, Add, Sub, Neg, MulC, ModC, Min, Max, SegIdx, SegStartAt,
                SegEndAt };
struct Expr;
using EP = std::shared_ptr<Expr>;
struct Expr {
  EK k;
  long long v = 0;
  EP a, b;
};
EP mk(EK k, EP a = nullptr, EP b = nullptr, long long v = 0) {
  auto e = std::make_shared<Expr>();
  e->k = k;
  e->a = a;
  e->b = b;
  e->v = v;
  return e;
}

enum class BK { True, False, And, Or, Not, Cmp };
struct BExpr;
using BP = std::shared_ptr<BExpr>;
struct BExpr {
  BK k;
  int op = 0;
  EP l, r;
  BP a, b;
};
BP mkb(BK k, BP a = nullptr, BP b = nullptr) {
  auto e = std::make_shared<BExpr>();
  e->k = k;
  e->a = a;
  e->b = b;
  return e;
}
BP mkcmp(int op, EP l, EP r) {
  auto e = mkb(BK::Cmp);
  e->op = op;
  e->l = l;
  e->r = r;
  return e;
}

bool contains_j(const EP& e) {
  if (!e) return false;
  if (e->k == EK::J) return true;
  return contains_j(e->a) || contains_j(e->b);
}
bool bcontains_j(const BP& b) {
  if (!b) return false;
  if (b->k == BK::Cmp) return contains_j(b->l) || contains_j(b->r);
  return bcontains_j(b->a) || bcontains_j(b->b);
}

// ---------------------------------------------------------------------------------------------
// parser
// ---------------------------------------------------------------------------------------------
struct Parser {
  std::vector<Tok> toks;
  size_t p = 0;
  int lineno = 0;

  const Tok& peek() const { return toks[p]; }
  [[noreturn]] void fail(const std::string& m) const {
    throw CompileError("line " + std::to_string(lineno) + ", col " + std::to_string(peek().col) +
                       ": " + m);
  }
  bool accept(T t) {
    if (peek().t == t) { ++p; return true; }
    return false;
  }
  void expect(T t, const char* what) {
    if (!accept(t)) fail(std::string("expected ") + what);
  }

  EP primary() {
    const Tok& k = peek();
    if (accept(T::Int)) return mk(EK::Const, nullptr, nullptr, k.v);
    if (accept(T::Minus)) return mk(EK::Neg, primary());
    if (accept(T::LParen)) {
      EP e = arith();
      expect(T::RParen, "')'");
      return e;
    }
    if (k.t == T::Ident) {
      const std::string name = k.s;
      ++p;
      if (name == "i") return mk(EK::I);
      if (name == "j") return mk(EK::J);
      if (name == "S") return mk(EK::S);
      if (name == "nseg") return mk(EK::Nseg);
      auto args = [&](int n) {
        expect(T::LParen, "'('");
        std::vector<EP> v;
        v.push_back(arith());
        for (int q = 1; q < n; ++q) {
          expect(T::Comma, "','");
          v.push_back(arith());
        }
        expect(T::RParen, "')'");
        return v;
      };
      if (name == "min" || name == "max") {
        auto v = args(2);
        return mk(name == "min" ? EK::Min : EK::Max, v[0], v[1]);
      }
      if (name == "seg_idx") return mk(EK::SegIdx, args(1)[0]);
      if (name == "seg_start_at") return mk(EK::SegStartAt, args(1)[0]);
      if (name == "seg_end_at") return mk(EK::SegEndAt, args(1)[0]);
      if (name == "seg_start") return mk(EK::SegStartAt, mk(EK::SegIdx, args(1)[0]));
      if (name == "seg_end") return mk(EK::SegEndAt, mk(EK::SegIdx, args(1)[0]));
      --p;
      fail("unknown name '" + name + "'");
    }
    fail("expected an integer term");
  }
  EP term() {
    EP e = primary();
    while (peek().t == T::Star || peek().t == T::Percent) {
      const bool mod = peek().t == T::Percent;
      ++p;
      EP r = primary();
      if (mod) {
        if (r->k != EK::Const || r->v < 1) fail("'%' needs a positive constant divisor");
        e = mk(EK::ModC, e, nullptr, r->v);
      } else if (r->k == EK::Const) {
        e = mk(EK::MulC, e, nullptr, r->v);
      } else if (e->k == EK::Const) {
        e = mk(EK::MulC, r, nullptr, e->v);
      } else {
        fail("multiplication needs a constant factor");
      }
    }
    return e;
  }
  EP arith() {
    EP e = term();
    while (peek().t == T::Plus || peek().t == T::Minus) {
      const bool plus = peek().t == T::Plus;
      ++p;
      EP r = term();
      e = mk(plus ? EK::Add : EK::Sub, e, r);
    }
    return e;
  }
  static int relop(T t) {
    switch (t) {
      case T::Lt: return CMP_LT;
      case T::Le: return CMP_LE;
      case T::Gt: return CMP_GT;
      case T::Ge: return CMP_GE;
      case T::Eq: return CMP_EQ;
      case T::Ne: return CMP_NE;
      default: return -1;
    }
  }
  BP comparison() {
    EP l = arith();
    const int op = relop(peek().t);
    if (op < 0) fail("expected a comparison operator");
    ++p;
    EP r = arith();
    if (relop(peek().t) >= 0) fail("chained comparisons are not supported");
    return mkcmp(op, l, r);
  }
  BP bfactor() {
    if (accept(T::Not)) return mkb(BK::Not, bfactor());
    if (peek().t == T::Ident && peek().s == "true") { ++p; return mkb(BK::True); }
    if (peek().t == T::Ident && peek().s == "false") { ++p; return mkb(BK::False); }
    if (peek().t == T::LParen) {
      // either a parenthesised boolean or an arithmetic term starting a comparison
      const size_t save = p;
      try {
        return comparison();
      } catch (const CompileError&) {
        p = save;
      }
      ++p;
      BP b = bexpr();
      expect(T::RParen, "')'");
      return b;
    }
    return comparison();
  }
  BP bterm() {
    BP b = bfactor();
    while (accept(T::And)) b = mkb(BK::And, b, bfactor());
    return b;
  }
  BP bexpr() {
    BP b = bterm();
    while (accept(T::Or)) b = mkb(BK::Or, b, bterm());
    return b;
  }
};

// ---------------------------------------------------------------------------------------------
// linear normal form of integer terms
// ---------------------------------------------------------------------------------------------
struct Lin;
struct Atom {
  EK kind;                 // I, J, S, Nseg, Min, Max, ModC, SegIdx, SegStartAt, SegEndAt
  std::vector<Lin> args;
  long long c = 0;         // the divisor of ModC
  std::string key;
};
using AP = std::shared_ptr<Atom>;

struct Lin {
  long long c = 0;
  std::map<std::string, std::pair<long long, AP>> t;  // key -> (coefficient, atom)

  bool is_const() const { return t.empty(); }
  long long coef(const std::string& k) const {
    auto it = t.find(k);
    return it == t.end() ? 0 : it->second.first;
  }
  std::string str() const {
    std::string s;
    for (const auto& kv : t) {
      const long long a = kv.second.first;
      const std::string& key = kv.first;
      if (s.empty()) {
        if (a == 1) s = key;
        else if (a == -1) s = "-" + key;
        else s = std::to_string(a) + "*" + key;
      } else {
        if (a == 1) s += " + " + key;
        else if (a == -1) s += " - " + key;
        else if (a > 0) s += " + " + std::to_string(a) + "*" + key;
        else s += " - " + std::to_string(-a) + "*" + key;
      }
    }
    if (s.empty()) return std::to_string(c);
    if (c > 0) s += " + " + std::to_string(c);
    if (c < 0) s += " - " + std::to_string(-c);
    return s;
  }
};

Lin lconst(long long c) {
  Lin l;
  l.c = c;
  return l;
}
Lin latom(AP a) {
  Lin l;
  l.t[a->key] = {1, a};
  return l;
}
Lin ladd(const Lin& x, const Lin& y, long long sy = 1) {
  Lin r = x;
  r.c += sy * y.c;
  for (const auto& kv : y.t) {
    auto& slot = r.t[kv.first];
    if (!slot.second) slot.second = kv.second.second;
    slot.first += sy * kv.second.first;
    if (slot.first == 0) r.t.erase(kv.first);
  }
  return r;
}
Lin lscale(const Lin& x, long long k) {
  if (k == 0) return lconst(0);
  Lin r;
  r.c = x.c * k;
  for (const auto& kv : x.t) r.t[kv.first] = {kv.second.first * k, kv.second.second};
  return r;
}
bool lequal(const Lin& a, const Lin& b) { return a.str() == b.str(); }

AP make_atom(EK kind, std::vector<Lin> args, long long c = 0) {
  auto a = std::make_shared<Atom>();
  a->kind = kind;
  a->args = std::move(args);
  a->c = c;
  switch (kind) {
    case EK::ModC: a->key = "mod(" + a->args[0].str() + ", " + std::to_string(c) + ")"; break;
    case EK::I: a->key = "i"; break;
    case EK::J: a->key = "j"; break;
    case EK::S: a->key = "S"; break;
    case EK::Nseg: a->key = "nseg"; break;
    case EK::Min: a->key = "min(" + a->args[0].str() + ", " + a->args[1].str() + ")"; break;
    case EK::Max: a->key = "max(" + a->args[0].str() + ", " + a->args[1].str() + ")"; break;
    case EK::SegIdx: a->key = "seg_idx(" + a->args[0].str() + ")"; break;
    case EK::SegStartAt:
    case EK::SegEndAt: {
      const Lin& k = a->args[0];
      const bool plain = k.c == 0 && k.t.size() == 1 && k.t.begin()->second.first == 1 &&
                         k.t.begin()->second.second->kind == EK::SegIdx;
      const char* nm = kind == EK::SegStartAt ? "seg_start" : "seg_end";
      if (plain) a->key = std::string(nm) + "(" + k.t.begin()->second.second->args[0].str() + ")";
      else a->key = std::string(nm) + "_at(" + k.str() + ")";
      break;
    }
    default: throw CompileError("internal: bad atom");
  }
  return a;
}

Lin lin_of(const EP& e, bool allow_j) {
  switch (e->k) {
    case EK::Const: return lconst(e->v);
    case EK::I: case EK::S: case EK::Nseg: return latom(make_atom(e->k, {}));
    case EK::J:
      if (!allow_j) throw CompileError("j may appear only linearly, outside min/max/seg_* terms");
      return latom(make_atom(EK::J, {}));
    case EK::Add: return ladd(lin_of(e->a, allow_j), lin_of(e->b, allow_j));
    case EK::Sub: return ladd(lin_of(e->a, allow_j), lin_of(e->b, allow_j), -1);
    case EK::Neg: return lscale(lin_of(e->a, allow_j), -1);
    case EK::MulC: return lscale(lin_of(e->a, allow_j), e->v);
    case EK::Min: case EK::Max: {
      Lin x = lin_of(e->a, false), y = lin_of(e->b, false);
      if (x.is_const() && y.is_const())
        return lconst(e->k == EK::Min ? std::min(x.c, y.c) : std::max(x.c, y.c));
      if (lequal(x, y)) return x;
      Lin d = ladd(x, y, -1);
      if (d.is_const()) {  // x - y constant: the answer is known
        const bool x_small = d.c < 0;
        return (e->k == EK::Min) == x_small ? x : y;
      }
      if (x.str() > y.str()) std::swap(x, y);  // commutative: canonical argument order
      return latom(make_atom(e->k, {x, y}));
    }
    case EK::SegIdx: case EK::SegStartAt: case EK::SegEndAt:
      return latom(make_atom(e->k, {lin_of(e->a, false)}));
    case EK::ModC: {  // non-negative remainder by a positive constant
      Lin x = lin_of(e->a, false);
      if (x.is_const()) return lconst(((x.c % e->v) + e->v) % e->v);
      return latom(make_atom(EK::ModC, {x}, e->v));
    }
  }
  throw CompileError("internal: bad expression");
}

// ---------------------------------------------------------------------------------------------
// DNF
// ---------------------------------------------------------------------------------------------
struct Cmp {
  Lin diff;  // lhs - rhs
  int op;    // diff (op) 0
};
using Conj = std::vector<Cmp>;
using Dnf = std::vector<Conj>;
constexpr size_t kMaxConjuncts = 64;

int negate(int op) {
  switch (op) {
    case CMP_LT: return CMP_GE;
    case CMP_LE: return CMP_GT;
    case CMP_GT: return CMP_LE;
    case CMP_GE: return CMP_LT;
    case CMP_EQ: return CMP_NE;
    default: return CMP_EQ;
  }
}

Dnf dnf(const BP& b, bool neg) {
  switch (b->k) {
    case BK::True: return neg ? Dnf{} : Dnf{Conj{}};
    case BK::False: return neg ? Dnf{Conj{}} : Dnf{};
    case BK::Not: return dnf(b->a, !neg);
    case BK::And:
    case BK::Or: {
      const bool is_or = (b->k == BK::Or) != neg;  // De Morgan
      Dnf x = dnf(b->a, neg), y = dnf(b->b, neg);
      Dnf r;
      if (is_or) {
        r = x;
        r.insert(r.end(), y.begin(), y.end());
      } else {
        for (const auto& cx : x)
          for (const auto& cy : y) {
            Conj c = cx;
            c.insert(c.end(), cy.begin(), cy.end());
            r.push_back(c);
          }
      }
      if (r.size() > kMaxConjuncts) throw CompileError("rule expands to too many conjuncts");
      return r;
    }
    case BK::Cmp: {
      const int op = neg ? negate(b->op) : b->op;
      Lin d = ladd(lin_of(b->l, true), lin_of(b->r, true), -1);
      if (op == CMP_NE) return Dnf{Conj{Cmp{d, CMP_LT}}, Conj{Cmp{d, CMP_GT}}};
      return Dnf{Conj{Cmp{d, op}}};
    }
  }
  throw CompileError("internal: bad boolean");
}

bool eval_const_cmp(long long v, int op) {
  switch (op) {
    case CMP_LT: return v < 0;
    case CMP_LE: return v <= 0;
    case CMP_GT: return v > 0;
    case CMP_GE: return v >= 0;
    case CMP_EQ: return v == 0;
    default: return v != 0;
  }
}

// ---------------------------------------------------------------------------------------------
// interval extraction and canonicalisation
// ---------------------------------------------------------------------------------------------
struct Slot {
  std::vector<Cmp> conds;  // j-free comparisons, all must hold
  std::vector<Lin> lows;   // lo = max(lows) (0 if none)
  std::vector<Lin> highs;  // hi = min(highs) (S if none)
};

const char* op_str(int op) {
  static const char* s[] = {"<", "<=", ">", ">=", "==", "!="};
  return s[op];
}
std::string cmp_str(const Cmp& c) { return c.diff.str() + " " + op_str(c.op) + " 0"; }

void add_unique(std::vector<Lin>& v, const Lin& x) {
  for (const auto& y : v)
    if (lequal(x, y)) return;
  v.push_back(x);
}

// returns false if the conjunct is provably empty
bool extract(const Conj& conj, Slot& s) {
  for (const Cmp& c : conj) {
    const long long cj = c.diff.coef("j");
    Lin rest = c.diff;
    rest.t.erase("j");
    if (cj == 0) {
      if (rest.is_const()) {
        if (!eval_const_cmp(rest.c, c.op)) return false;
        continue;
      }
      bool dup = false;
      for (const auto& x : s.conds)
        if (x.op == c.op && lequal(x.diff, rest)) dup = true;
      if (!dup) s.conds.push_back(Cmp{rest, c.op});
      continue;
    }
    if (cj != 1 && cj != -1) throw CompileError("j must appear with coefficient +1 or -1");
    // j*cj + rest (op) 0  ->  j (op') X
    int op = c.op;
    Lin X = lscale(rest, -1);
    if (cj == -1) {
      X = rest;
      switch (op) {
        case CMP_LT: op = CMP_GT; break;
        case CMP_LE: op = CMP_GE; break;
        case CMP_GT: op = CMP_LT; break;
        case CMP_GE: op = CMP_LE; break;
        default: break;
      }
    }
    switch (op) {
      case CMP_LT: add_unique(s.highs, X); break;
      case CMP_LE: add_unique(s.highs, ladd(X, lconst(1))); break;
      case CMP_GT: add_unique(s.lows, ladd(X, lconst(1))); break;
      case CMP_GE: add_unique(s.lows, X); break;
      case CMP_EQ:
        add_unique(s.lows, X);
        add_unique(s.highs, ladd(X, lconst(1)));
        break;
      default: throw CompileError("internal: != after DNF");
    }
  }
  // a bound that another bound dominates by a constant is redundant
  auto prune = [](std::vector<Lin>& v, bool keep_smaller) {
    std::vector<Lin> out;
    for (size_t a = 0; a < v.size(); ++a) {
      bool redundant = false;
      for (size_t b = 0; b < v.size() && !redundant; ++b) {
        if (a == b) continue;
        Lin d = ladd(v[a], v[b], -1);  // v[a] - v[b]
        if (!d.is_const()) continue;
        redundant = keep_smaller ? (d.c > 0 || (d.c == 0 && b < a)) : (d.c < 0 || (d.c == 0 && b < a));
      }
      if (!redundant) out.push_back(v[a]);
    }
    v = out;
  };
  prune(s.highs, true);
  prune(s.lows, false);
  // provably empty: some upper bound minus some lower bound is a constant <= 0
  for (const auto& h : s.highs) {
    if (h.is_const() && h.c <= 0) return false;
    for (const auto& l : s.lows) {
      Lin d = ladd(h, l, -1);
      if (d.is_const() && d.c <= 0) return false;
    }
  }
  return true;
}

std::string slot_key(const Slot& s) {
  std::vector<std::string> c, l, h;
  for (const auto& x : s.conds) c.push_back(cmp_str(x));
  for (const auto& x : s.lows) l.push_back(x.str());
  for (const auto& x : s.highs) h.push_back(x.str());
  std::sort(c.begin(), c.end());
  std::sort(l.begin(), l.end());
  std::sort(h.begin(), h.end());
  std::string k;
  for (auto& x : c) k += x + ";";
  k += "|";
  for (auto& x : l) k += x + ";";
  k += "|";
  for (auto& x : h) k += x + ";";
  return k;
}

// ---------------------------------------------------------------------------------------------
// code emission
// ---------------------------------------------------------------------------------------------
struct Emitter {
  std::vector<int32_t> code;
  void op(int32_t o) { code.push_back(o); }
  void op(int32_t o, long long imm) {
    if (imm < INT32_MIN || imm > INT32_MAX) throw CompileError("constant out of int32 range");
    code.push_back(o);
    code.push_back(static_cast<int32_t>(imm));
  }
  void atom(const Atom& a) {
    switch (a.kind) {
      case EK::I: op(OP_I); break;
      case EK::S: op(OP_S); break;
      case EK::Nseg: op(OP_NSEG); break;
      case EK::Min: lin(a.args[0]); lin(a.args[1]); op(OP_MIN); break;
      case EK::Max: lin(a.args[0]); lin(a.args[1]); op(OP_MAX); break;
      case EK::SegIdx: {
        // seg_idx(i) is the common case: the evaluator computes it once per row
        const Lin& x = a.args[0];
        const bool row_itself = x.c == 0 && x.t.size() == 1 && x.t.begin()->second.first == 1 &&
                                x.t.begin()->second.second->kind == EK::I;
        if (row_itself) {
          op(OP_SEG_IDX_I);
        } else {
          lin(x);
          op(OP_SEG_IDX);
        }
        break;
      }
      case EK::SegStartAt: lin(a.args[0]); op(OP_SEG_START_AT); break;
      case EK::SegEndAt: lin(a.args[0]); op(OP_SEG_END_AT); break;
      case EK::ModC: lin(a.args[0]); op(OP_MODC, a.c); break;
      default: throw CompileError("internal: j in an endpoint");
    }
  }
  void lin(const Lin& l) {
    bool first = true;
    for (const auto& kv : l.t) {
      atom(*kv.second.second);
      if (kv.second.first != 1) op(OP_MULC, kv.second.first);
      if (!first) op(OP_ADD);
      first = false;
    }
    if (first) op(OP_CONST, l.c);
    else if (l.c != 0) { op(OP_CONST, l.c); op(OP_ADD); }
  }
  void expr(const EP& e) { lin(lin_of(e, false)); }
  void boolean(const BP& b) {
    switch (b->k) {
      case BK::True: op(OP_CONST, 1); break;
      case BK::False: op(OP_CONST, 0); break;
      case BK::Not: boolean(b->a); op(OP_NOT); break;
      case BK::And: boolean(b->a); boolean(b->b); op(OP_AND); break;
      case BK::Or: boolean(b->a); boolean(b->b); op(OP_OR); break;
      case BK::Cmp: expr(b->l); expr(b->r); op(OP_CMP, b->op); break;
    }
  }
  int16_t begin() { return static_cast<int16_t>(code.size()); }
  void end() { op(OP_END); }
};

// stack depth needed by a program (the kernel's evaluator holds kMaxStack entries)
int max_depth(const std::vector<int32_t>& code, int start) {
  int d = 0, m = 0;
  for (size_t p = static_cast<size_t>(start); p < code.size(); ++p) {
    switch (code[p]) {
      case OP_END: return m;
      case OP_CONST: ++d; ++p; break;
      case OP_I: case OP_S: case OP_NSEG: case OP_SEG_IDX_I: ++d; break;
      case OP_ADD: case OP_SUB: case OP_MIN: case OP_MAX: case OP_AND: case OP_OR: --d; break;
      case OP_CMP: --d; ++p; break;
      case OP_MULC: case OP_MODC: ++p; break;
      default: break;  // unary ops keep the depth
    }
    m = std::max(m, d);
  }
  return m;
}

// ---- the same endpoints as CUDA C++ (the mask-specific kernel's row evaluator) --------------
// Names in scope of the generated code: i (row), ki (= seg_idx(i)), seg (segment starts in shared
// memory), nseg, S.  Sums and products wrap like the stack programs' arithmetic.
std::string c_lin(const Lin& l);
std::string c_const(long long v);
std::string c_atom(const Atom& a) {
  switch (a.kind) {
    case EK::I: return "i";
    case EK::S: return "S";
    case EK::Nseg: return "nseg";
    case EK::Min: return "cmcore::imin(" + c_lin(a.args[0]) + ", " + c_lin(a.args[1]) + ")";
    case EK::Max: return "cmcore::imax(" + c_lin(a.args[0]) + ", " + c_lin(a.args[1]) + ")";
    case EK::SegIdx: {
      const Lin& x = a.args[0];
      const bool row_itself = x.c == 0 && x.t.size() == 1 && x.t.begin()->second.first == 1 &&
                              x.t.begin()->second.second->kind == EK::I;
      return row_itself ? "ki" : "cmcore::seg_index(seg, nseg, " + c_lin(x) + ")";
    }
    case EK::SegStartAt: return "cmcore::seg_start_at(seg, nseg, " + c_lin(a.args[0]) + ")";
    case EK::SegEndAt: return "cmcore::seg_end_at(seg, nseg, " + c_lin(a.args[0]) + ")";
    case EK::ModC: return "cmcore::imod(" + c_lin(a.args[0]) + ", " + c_const(a.c) + ")";
    default: throw CompileError("internal: j in an endpoint");
  }
}
std::string c_const(long long v) {
  if (v < INT32_MIN || v > INT32_MAX) throw CompileError("constant out of int32 range");
  return "(" + std::to_string(v) + ")";
}
std::string c_lin(const Lin& l) {
  std::string acc;
  for (const auto& kv : l.t) {
    std::string term = c_atom(*kv.second.second);
    if (kv.second.first != 1) term = "cmcore::wmul(" + term + ", " + c_const(kv.second.first) + ")";
    acc = acc.empty() ? term : "cmcore::wadd(" + acc + ", " + term + ")";
  }
  if (acc.empty()) return c_const(l.c);
  if (l.c != 0) acc = "cmcore::wadd(" + acc + ", " + c_const(l.c) + ")";
  return acc;
}
const char* c_op(int op) {
  static const char* s[] = {"<", "<=", ">", ">=", "==", "!="};
  return s[op];
}
std::string c_bool(const BP& b) {
  switch (b->k) {
    case BK::True: return "true";
    case BK::False: return "false";
    case BK::Not: return "!(" + c_bool(b->a) + ")";
    case BK::And: return "(" + c_bool(b->a) + " && " + c_bool(b->b) + ")";
    case BK::Or: return "(" + c_bool(b->a) + " || " + c_bool(b->b) + ")";
    case BK::Cmp:
      return "(" + c_lin(lin_of(b->l, false)) + " " + c_op(b->op) + " " +
             c_lin(lin_of(b->r, false)) + ")";
  }
  return "false";
}

std::string bstr(const BP& b) {
  switch (b->k) {
    case BK::True: return "all";
    case BK::False: return "false";
    case BK::Not: return "!(" + bstr(b->a) + ")";
    case BK::And: return "(" + bstr(b->a) + " && " + bstr(b->b) + ")";
    case BK::Or: return "(" + bstr(b->a) + " || " + bstr(b->b) + ")";
    case BK::Cmp:
      return lin_of(b->l, true).str() + " " + op_str(b->op) + " " + lin_of(b->r, true).str();
  }
  return "?";
}

}  // namespace

// ---------------------------------------------------------------------------------------------
// the compiled spec
// ---------------------------------------------------------------------------------------------
// The mask-specific kernel of one (forward, backward) pair, compiled and loaded once, on first use.
struct PairKernel {
  uint64_t bwd_serial = 0;
  const void* kernel = nullptr;
  int rc = CM_OK;          // why kernel is null, if it is
  std::string log;
};

struct SpecImpl {
  DevProg prog;
  uint64_t serial = 0;     // identifies the spec in the pair cache of other specs
  std::string text;        // describe() output
  std::string gen;         // body of the row evaluator of the mask-specific kernel (CUDA C++)
  std::mutex mu;           // guards `pairs`
  std::list<PairKernel> pairs;  // kernels with this spec as the forward one (stable addresses)
};

std::atomic<uint64_t> g_spec_serial{1};

// CUDA C++ of a row evaluator struct named `name`.
std::string evaluator_source(const SpecImpl& s, const std::string& name) {
  return "struct " + name + " {\n"
         "  __device__ __forceinline__ void row(int i, int ki, const int* seg, int nseg, int S,\n"
         "                                      int* lo, int* hi) const {\n"
         "    (void)i; (void)ki; (void)seg; (void)nseg; (void)S; (void)lo; (void)hi;\n" +
         s.gen + "  }\n};\n";
}

// Source of the mask-specific preprocess kernel of a (forward, backward) pair of specs: the two
// row evaluators and the shared kernel body, one launch for both halves of the descriptor.
std::string pair_source(const SpecImpl& f, const SpecImpl& b) {
  return "// Mask-specific preprocess kernel generated from a forward and a backward MaskSpec.\n"
         "#include \"descriptor_core.cuh\"\n" +
         evaluator_source(f, "EvalFwd") + evaluator_source(b, "EvalBwd") +
         "extern \"C\" __global__ void __launch_bounds__(cmcore::kThreads)\n"
         "cm_generated_descriptor(const __grid_constant__ cmcore::DescCore p) {\n"
         "  cmcore::descriptor_kernel<" + std::to_string(f.prog.ni) + ", " +
         std::to_string(b.prog.ni) + ">(p, EvalFwd(), EvalBwd());\n"
         "}\n";
}

static int compile(const char* text, SpecImpl& out) {
  std::istringstream in(text);
  std::string line;
  int lineno = 0;
  Emitter em;
  DevProg& P = out.prog;
  std::memset(&P, 0, sizeof(P));
  std::ostringstream desc;
  std::ostringstream gen;  // body of the generated row evaluator
  int ni = 0, nreg = 0;
  while (std::getline(in, line)) {
    ++lineno;
    const size_t hash = line.find('#');
    if (hash != std::string::npos) line = line.substr(0, hash);
    bool blank = true;
    for (char c : line)
      if (!std::isspace(static_cast<unsigned char>(c))) blank = false;
    if (blank) continue;
    Parser ps;
    ps.toks = lex(line, lineno);
    ps.lineno = lineno;
    if (!(ps.peek().t == T::Ident && ps.peek().s == "region")) ps.fail("expected 'region'");
    ++ps.p;
    BP guard;
    if (ps.peek().t == T::Ident && ps.peek().s == "all" && ps.toks[ps.p + 1].t == T::Colon) {
      ++ps.p;
      guard = mkb(BK::True);
    } else {
      guard = ps.bexpr();
    }
    ps.expect(T::Colon, "':' between guard and rule");
    BP rule = ps.bexpr();
    if (ps.peek().t != T::End) ps.fail("unexpected text after the rule");
    if (bcontains_j(guard)) ps.fail("a Region guard may use i only, not j");
    if (nreg >= kMaxRegions) ps.fail("too many Regions");

    // lower the rule
    Dnf d = dnf(rule, false);
    std::vector<Slot> slots;
    std::vector<std::string> keys;
    for (const Conj& c : d) {
      Slot s;
      if (!extract(c, s)) continue;
      const std::string k = slot_key(s);
      bool dup = false;
      for (const auto& x : keys)
        if (x == k) dup = true;
      if (dup) continue;
      keys.push_back(k);
      slots.push_back(s);
    }
    if (static_cast<int>(slots.size()) > kMaxSlots)
      throw CompileError("line " + std::to_string(lineno) + ": rule needs " +
                         std::to_string(slots.size()) + " intervals (limit " +
                         std::to_string(kMaxSlots) + ")");
    const int r = nreg++;
    ni = std::max(ni, static_cast<int>(slots.size()));
    P.guard[r] = em.begin();
    em.boolean(guard);
    em.end();
    P.nslot[r] = static_cast<int16_t>(slots.size());
    desc << "region " << r << " when " << bstr(guard) << "\n";
    gen << "    if (" << c_bool(guard) << ") {\n";
    for (size_t n = 0; n < slots.size(); ++n) {
      const Slot& s = slots[n];
      if (s.conds.empty()) {
        P.cond[r][n] = -1;
      } else {
        P.cond[r][n] = em.begin();
        for (size_t q = 0; q < s.conds.size(); ++q) {
          em.lin(s.conds[q].diff);
          em.op(OP_CONST, 0);
          em.op(OP_CMP, s.conds[q].op);
          if (q) em.op(OP_AND);
        }
        em.end();
      }
      std::string lo_s, hi_s;
      P.lo[r][n] = em.begin();
      if (s.lows.empty()) { em.op(OP_CONST, 0); lo_s = "0"; }
      for (size_t q = 0; q < s.lows.size(); ++q) {
        em.lin(s.lows[q]);
        if (q) em.op(OP_MAX);
        lo_s = q ? "max(" + lo_s + ", " + s.lows[q].str() + ")" : s.lows[q].str();
      }
      em.end();
      P.hi[r][n] = em.begin();
      if (s.highs.empty()) { em.op(OP_S); hi_s = "S"; }
      for (size_t q = 0; q < s.highs.size(); ++q) {
        em.lin(s.highs[q]);
        if (q) em.op(OP_MIN);
        hi_s = q ? "min(" + hi_s + ", " + s.highs[q].str() + ")" : s.highs[q].str();
      }
      em.end();
      std::string lo_c = c_const(0), hi_c = "S", cond_c;
      for (size_t q = 0; q < s.lows.size(); ++q)
        lo_c = q ? "cmcore::imax(" + lo_c + ", " + c_lin(s.lows[q]) + ")" : c_lin(s.lows[q]);
      for (size_t q = 0; q < s.highs.size(); ++q)
        hi_c = q ? "cmcore::imin(" + hi_c + ", " + c_lin(s.highs[q]) + ")" : c_lin(s.highs[q]);
      for (size_t q = 0; q < s.conds.size(); ++q)
        cond_c += std::string(q ? " && " : "") + "(" + c_lin(s.conds[q].diff) + " " +
                  c_op(s.conds[q].op) + " 0)";
      const std::string ind = cond_c.empty() ? "      " : "        ";
      if (!cond_c.empty()) gen << "      if (" << cond_c << ") {\n";
      gen << ind << "lo[" << n << "] = " << lo_c << ";\n";
      gen << ind << "hi[" << n << "] = " << hi_c << ";\n";
      if (!cond_c.empty()) gen << "      }\n";
      desc << "  slot " << n << ": [" << lo_s << ", " << hi_s << ")";
      for (size_t q = 0; q < s.conds.size(); ++q)
        desc << (q ? " and " : " if ") << cmp_str(s.conds[q]);
      desc << "\n";
    }
    gen << "      return;\n    }\n";
    if (em.code.size() > static_cast<size_t>(kMaxCode))
      throw CompileError("spec too large (endpoint programs exceed " + std::to_string(kMaxCode) +
                         " words)");
  }
  if (nreg == 0) throw CompileError("spec has no region");
  // programs must fit the device evaluator's stack
  for (int r = 0; r < nreg; ++r) {
    int m = max_depth(em.code, P.guard[r]);
    for (int n = 0; n < P.nslot[r]; ++n) {
      if (P.cond[r][n] >= 0) m = std::max(m, max_depth(em.code, P.cond[r][n]));
      m = std::max(m, max_depth(em.code, P.lo[r][n]));
      m = std::max(m, max_depth(em.code, P.hi[r][n]));
    }
    if (m > kMaxStack) throw CompileError("expression nesting too deep");
  }
  P.ni = std::max(ni, 1);
  P.nreg = nreg;
  for (size_t q = 0; q < em.code.size(); ++q) P.code[q] = em.code[q];
  out.text = "intervals " + std::to_string(P.ni) + "\n" + desc.str();
  out.gen = gen.str();
  out.serial = g_spec_serial.fetch_add(1);
  return CM_OK;
}

const DevProg* spec_program(const cm_spec* s);
const void* pair_generated_kernel(const cm_spec* fwd, const cm_spec* bwd);
int compile_generated_kernel(const std::string& source, std::vector<char>* cubin, std::string* log);
int load_generated_kernel(const std::string& source, const void** kernel, std::string* log);

}  // namespace cm

struct cm_spec {
  cm::SpecImpl impl;
};

const cm::DevProg* cm::spec_program(const cm_spec* s) { return &s->impl.prog; }

// The pair's entry in the forward spec's cache, compiled and loaded on first use.
static const cm::PairKernel& pair_kernel(const cm_spec* fwd, const cm_spec* bwd) {
  cm::SpecImpl& im = const_cast<cm_spec*>(fwd)->impl;
  std::lock_guard<std::mutex> lock(im.mu);
  for (const cm::PairKernel& e : im.pairs)
    if (e.bwd_serial == bwd->impl.serial) return e;
  im.pairs.emplace_back();
  cm::PairKernel& e = im.pairs.back();
  e.bwd_serial = bwd->impl.serial;
  e.rc = cm::load_generated_kernel(cm::pair_source(fwd->impl, bwd->impl), &e.kernel, &e.log);
  return e;
}

const void* cm::pair_generated_kernel(const cm_spec* fwd, const cm_spec* bwd) {
  return pair_kernel(fwd, bwd).kernel;
}

extern "C" {

CM_API int cm_compile_spec(const char* text, cm_spec** out, char* err, size_t err_len) {
  if (err && err_len) err[0] = 0;
  if (!text || !out) return CM_ERR_INVALID_ARG;
  *out = nullptr;
  auto* s = new cm_spec();
  try {
    cm::compile(text, s->impl);
  } catch (const std::exception& e) {
    if (err && err_len) std::snprintf(err, err_len, "%s", e.what());
    delete s;
    return CM_ERR_PARSE;
  }
  *out = s;
  return CM_OK;
}

CM_API void cm_spec_free(cm_spec* spec) { delete spec; }

CM_API int cm_spec_num_intervals(const cm_spec* spec, int* ni_max) {
  if (!spec || !ni_max) return CM_ERR_INVALID_ARG;
  *ni_max = spec->impl.prog.ni;
  return CM_OK;
}

CM_API int cm_descriptor_kernel_source(const cm_spec* fwd, const cm_spec* bwd, char* buf,
                                       size_t len, size_t* needed) {
  if (!fwd || !bwd) return CM_ERR_INVALID_ARG;
  const std::string t = cm::pair_source(fwd->impl, bwd->impl);
  if (needed) *needed = t.size() + 1;
  if (buf && len) std::snprintf(buf, len, "%s", t.c_str());
  return CM_OK;
}

CM_API int cm_descriptor_kernel_status(const cm_spec* fwd, const cm_spec* bwd, int load, char* log,
                                       size_t log_len) {
  if (log && log_len) log[0] = 0;
  if (!fwd || !bwd) return CM_ERR_INVALID_ARG;
  int rc;
  std::string text;
  if (load) {
    const cm::PairKernel& e = pair_kernel(fwd, bwd);
    rc = e.rc;
    text = e.log;
  } else {
    std::vector<char> cubin;
    rc = cm::compile_generated_kernel(cm::pair_source(fwd->impl, bwd->impl), &cubin, &text);
  }
  if (log && log_len) std::snprintf(log, log_len, "%s", text.c_str());
  return rc;
}

CM_API int cm_spec_kernel_source(const cm_spec* spec, char* buf, size_t len, size_t* needed) {
  return cm_descriptor_kernel_source(spec, spec, buf, len, needed);
}

CM_API int cm_spec_kernel_status(const cm_spec* spec, int load, char* log, size_t log_len) {
  return cm_descriptor_kernel_status(spec, spec, load, log, log_len);
}

CM_API int cm_spec_describe(const cm_spec* spec, char* buf, size_t len, size_t* needed) {
  if (!spec) return CM_ERR_INVALID_ARG;
  const std::string& t = spec->impl.text;
  if (needed) *needed = t.size() + 1;
  if (buf && len) std::snprintf(buf, len, "%s", t.c_str());
  return CM_OK;
}

}  // extern "C"

// Endpoint programs: the compiled form of a MaskSpec that the preprocess kernel evaluates.
//
// CompileMask lowers each Region's visibility rule offline to symbolic interval endpoints
// (section 3.2.2) and evaluates them online against batch metadata (section 3.3).  Here the
// lowered endpoints are small stack programs over int32: one guard program per Region, and per
// slot an optional condition program plus the `lo` and `hi` endpoint programs.  A row takes the
// first Region whose guard holds; slot n of that Region gives the half-open interval
// [lo, hi) of the other index, or (0, 0) when its condition fails or the interval is empty.
#pragma once
#include <cstdint>

namespace cm {

constexpr int kMaxRegions = 8;
constexpr int kMaxSlots = 8;
constexpr int kMaxCode = 448;
constexpr int kMaxStack = 16;

enum Op : int32_t {
  OP_END = 0,
  OP_CONST = 1,       // imm
  OP_I = 2,           // the row index
  OP_S = 3,           // sequence length
  OP_NSEG = 4,        // segment count of the sample
  OP_ADD = 5,
  OP_SUB = 6,
  OP_MULC = 7,        // imm
  OP_MIN = 8,
  OP_MAX = 9,
  OP_SEG_IDX = 10,    // segment holding position e (clamped to [0, nseg-1])
  OP_SEG_START_AT = 11,  // seg[clamp(k, 0, nseg)]
  OP_SEG_END_AT = 12,    // seg[clamp(k + 1, 0, nseg)]
  OP_CMP = 13,        // imm = CmpOp; pops b, a; pushes (a op b)
  OP_AND = 14,
  OP_OR = 15,
  OP_NOT = 16,
  OP_NEG = 17,
  OP_SEG_IDX_I = 18,  // seg_idx(i) of the row, computed once per row by the evaluator
  OP_MODC = 19,       // imm > 0: non-negative remainder
};

enum CmpOp : int32_t { CMP_LT = 0, CMP_LE = 1, CMP_GT = 2, CMP_GE = 3, CMP_EQ = 4, CMP_NE = 5 };

// Passed by value as a kernel parameter (one per spec).
struct DevProg {
  int32_t ni;        // slots per row (compiler-derived interval count)
  int32_t nreg;      // number of Regions
  int16_t guard[kMaxRegions];
  int16_t nslot[kMaxRegions];
  int16_t cond[kMaxRegions][kMaxSlots];  // -1: no condition
  int16_t lo[kMaxRegions][kMaxSlots];
  int16_t hi[kMaxRegions][kMaxSlots];
  int32_t code[kMaxCode];
};

}  // namespace cm

// Descriptor-guided attention, forward (CompileMask section 3.3.2), for sm_103a.
//
// One CTA computes one 128-row query tile of one (sample, head).  The Tile-State Bitmap row of
// that query tile lists the key tiles to visit: empty tiles are skipped, full tiles run without
// any mask, and partial tiles check every score against the row's visible intervals with one
// unsigned subtraction and one comparison per interval (section 4.4), replacing invisible scores
// with -inf before the online softmax.
//
// Each 128-key tile is split into two column halves that keep separate online-softmax states:
// half h has its own running max and row sum per query row and its own output accumulator
// O_h += P_h V_h (P_h: the half's 64 keys, V_h: the matching 64 rows of V).  The two states are
// merged once, at the end: O = (O_0 2^(m_0 - M) + O_1 2^(m_1 - M)) / (l_0 2^(m_0 - M) +
// l_1 2^(m_1 - M)) with M = max(m_0, m_1).  So the two warps that share a query row never wait
// for each other inside the loop.
//
// Warp roles (320 threads):
//   warps 0-7  softmax.  Warp w serves TMEM lane quarter w % 4 (query rows 32*(w%4) ..) and
//              column half w / 4 of each S tile.  It reads its 64 scores per row from TMEM,
//              masks partial tiles, runs its half's online softmax in the log2 domain, writes P
//              (bf16 pairs) back over the S columns it has read, rescales its half's O when the
//              running max moved, and at the end merges the halves and writes O and the LSE.
//   warp 8     TMA producer: Q once, then K and V of each visited key tile into one of 3 stages
//              (one barrier for both tiles; the stage frees when the tile's PV MMAs completed).
//   warps 9-10 MMA issuers, one thread each: the thread of warp 9 + t issues the MMAs of the key
//              tiles n with n % 2 == t: S(n) = Q K(n)^T (Q and K from shared memory) and, per
//              half, O_h += P_h(n) V_h(n) with P_h read from TMEM.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O_0 [256, 256+d), O_1 [384, 384+d).  P of tile n
// lives in S buffer n % 2: keys [0,64) in columns [0,32), keys [64,128) in [64,96).
// Why two issuers: a thread that issues tcgen05 MMAs stalls on every barrier wait (even on a phase
// that is already complete), and the tensor pipe holds too few queued 128 x 128 MMAs to cover
// the stall, so a single issuer leaves a gap in the pipe at each wait.  With the tiles dealt by
// parity, one thread's MMAs run while the other waits.
// Ordering: a thread issues S(n+2) into a buffer right after PV(n), which reads P(n) from that
// buffer (tcgen05 MMAs of one thread run in issue order).  PV(n) accumulates into the O_h that
// PV(n-1) of the other thread updates, so it is issued only after PV(n-1) has completed (the
// stage barrier of tile n-1): the accumulations never overlap.
// The softmax warps wait for PV(n-1) (its stage's release) only when they must rescale O: the
// completion of S(n), which they wait for anyway, already covers every PV issued before it (up to
// PV(n-2)).
// The running max is refreshed lazily: O and l are rescaled only when the row max grows by more
// than 2^8, which keeps P <= 256 and the result exact because O, l and the LSE use the same max.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "kernels.h"
#include "mask.cuh"
#include "ptx.cuh"
#include "tma_host.h"

namespace cm {
namespace fwd {

constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;   // and 10
constexpr int kThreads = 352;
constexpr int kStages = 3;  // K ring and V ring depth

constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;  // O_h at kColO + 128 * h

template <int D>
struct Smem {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kQ = 0;  // also the merge exchange area once every MMA is done
  static constexpr uint32_t kKV = kTileBytes;  // stage s: K at kKV + 2*s*tile, V right after it
  static constexpr uint32_t kBar = kKV + kStages * 2u * kTileBytes;
  static constexpr uint32_t kRow = kBar + 256u;  // bitmap row: at most 64 words (NT <= 1024)
  static constexpr uint32_t kTotal = kRow + 256u;
  static constexpr uint32_t kAlloc = kTotal + 1024u;  // slack for 1024-byte alignment
};
static_assert(Smem<128>::kAlloc <= 232448, "forward shared memory exceeds 227 KB");

enum {
  B_Q = 0,        // Q tile in shared memory (TMA)
  B_KVFULL = 1,   // +stage: K and V of a key tile landed (TMA, 2 tiles of bytes)
  B_KVEMPTY = 4,  // +stage: S and PV of the stage's tile have completed (also "O is up to date",
                  // and the other issuer's go-ahead for the next PV)
  B_SFULL = 7,    // +buffer
  B_PFULL = 9,    // +buffer: P of a tile in that S buffer, both halves (8 arrivals)
  B_PAIR = 11,    // +quarter: merge exchange of a warp pair (2 arrivals, once)
  B_ALLDONE = 15, // every MMA of the CTA has completed (once; one commit per issuer)
  B_DRAIN = 16,   // +issuer, abort path only: every MMA the issuer issued so far has completed
  B_COUNT = 18
};

template <int D, int MAXNI>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  using L = Smem<D>;
  constexpr int kHalf = D / 2;  // output columns per softmax warp in the merge
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * B_COUNT + 4);
  int* s_ntiles = reinterpret_cast<int*>(smem + L::kBar + 8 * B_COUNT + 8);
  uint32_t* bmrow = reinterpret_cast<uint32_t*>(smem + L::kRow);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const WaitCtl wait{abort_flag, p.status, p.wait_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int item_idx, h;  // head-grouped chunks of the schedule (L2 locality, longest rows first)
  cta_work(blockIdx.x, p.B * p.NT, p.H, item_idx, h);
  const int item = p.sched[item_idx];
  const int b = item >> 16;
  const int qt = item & 0xFFFF;
  if (b < 0 || b >= p.B || qt >= p.NT) {  // a schedule entry that no descriptor build wrote
    if (threadIdx.x == 0) set_status(p.status, kDevBadSchedule, item_idx);
    return;
  }
  const int bh = b * p.H + h;

  // ---- set-up: barriers, bitmap row, TMEM ---------------------------------------------------
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KVFULL + s), 1);
      mbar_init(bar(B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), kSoftmaxWarps);
    }
    for (int s = 0; s < 4; ++s) mbar_init(bar(B_PAIR + s), 2);
    mbar_init(bar(B_ALLDONE), 2);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN + 1), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    // this CTA's bitmap row (W <= 64 words) and its count of non-empty key tiles
    const uint32_t* row = p.bm + (static_cast<size_t>(b) * p.NT + qt) * p.W;
    int cnt = 0;
    for (int w = lane; w < p.W; w += 32) {
      const uint32_t x = row[w];
      bmrow[w] = x;
      cnt += __popc((x | (x >> 1)) & 0x55555555u);
    }
    cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
    if (lane == 0) *s_ntiles = cnt;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nt = *s_ntiles;
  // asynchronous work issued so far, for the abort path: K/V stages armed (producer), any MMA
  // issued (MMA thread)
  int n_armed = 0;
  bool mma_issued = false;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int row0 = bh * p.S;
      mbar_arrive_expect_tx(bar(B_Q), L::kTileBytes);
      for (int x = 0; x < D / 64; ++x)
        tma_load_2d(sbase + L::kQ + x * 16384u, &tmQ, x * 64, row0 + qt * 128, bar(B_Q));
      int kt = next_tile(bmrow, p.NT, 0);
      for (int n = 0; n < nt; ++n, kt = next_tile(bmrow, p.NT, kt + 1)) {
        const int st = n % kStages;
        if (n >= kStages &&
            !wait(bar(B_KVEMPTY + st), ((n / kStages) - 1) & 1, 0x101))
          break;
        const uint32_t sK = sbase + L::kKV + st * 2u * L::kTileBytes;
        n_armed = n + 1;
        mbar_arrive_expect_tx(bar(B_KVFULL + st), 2u * L::kTileBytes);
        for (int x = 0; x < D / 64; ++x)
          tma_load_2d(sK + x * 16384u, &tmK, x * 64, row0 + kt * 128, bar(B_KVFULL + st));
        for (int x = 0; x < D / 64; ++x)
          tma_load_2d(sK + L::kTileBytes + x * 16384u, &tmV, x * 64, row0 + kt * 128,
                      bar(B_KVFULL + st));
      }
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ---------------------------------------------------------------- MMA issuers
    const int par = warp - kMmaWarp;  // this thread's key tiles: n % 2 == par
    if (lane == 0 && nt > par) {
      constexpr uint32_t idS = make_idesc_bf16(128, 128, 0, 0);  // A = Q, B = K, both K-major
      constexpr uint32_t idO = make_idesc_bf16(128, D, 0, 1);    // A = P (TMEM), B = V MN-major
      const uint32_t dQ = sdesc_lo(sbase + L::kQ, 16u);
      bool ok = wait(bar(B_Q), 0, 0x102);
      // O_h += P_h V_h for tile m: keys [64h, +64) are the K-steps kk = 4h .. 4h+3.  V(m) landed
      // before S(m) was issued (same barrier as K(m)).
      auto issue_pv = [&](int m) -> bool {
        const int st = m % kStages;
        // one barrier per S buffer: the softmax warps can be at most one tile ahead of this
        // wait, so a barrier never runs two phases ahead of its waiter
        if (!wait(bar(B_PFULL + (m & 1)), (m >> 1) & 1, 0x103))
          return false;
        // PV(m-1), issued by the other thread, has completed.  Its stage barrier cannot run a
        // phase ahead of this wait: PV(m+2) of that stage needs PV(m+1), which needs PV(m).
        if (m >= 1 &&
            !wait(bar(B_KVEMPTY + (m - 1) % kStages), ((m - 1) / kStages) & 1, 0x104))
          return false;
        tc_fence_after();
        const uint32_t dV = sdesc_lo(sbase + L::kKV + st * 2u * L::kTileBytes + L::kTileBytes, 16384u);
        const uint32_t sP = tmem + kColS + (m & 1) * 128;
        const uint32_t acc0 = m > 0 ? 1u : 0u;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * hh + k4;
            umma_ts_lo(tmem + kColO + 128 * hh, sP + 64 * hh + 8 * k4, dV + kstep_mnmajor(kk), idO,
                       k4 > 0 ? 1u : acc0);
          }
        }
        umma_commit(bar(B_KVEMPTY + st));
        return true;
      };
      // S(n) into buffer n % 2 = Q K(n)^T
      auto issue_s = [&](int n) -> bool {
        const int st = n % kStages;
        if (!wait(bar(B_KVFULL + st), (n / kStages) & 1, 0x105))
          return false;
        tc_fence_after();
        mma_issued = true;
        const uint32_t dK = sdesc_lo(sbase + L::kKV + st * 2u * L::kTileBytes, 16u);
        const uint32_t dS = tmem + kColS + (n & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_lo(dS, dQ + kstep_kmajor(kk), dK + kstep_kmajor(kk), idS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL + (n & 1)));
        return true;
      };
      // S(par) first; then per own tile n: PV(n) once P(n) is written and PV(n-1) is done, and
      // S(n+2) into the buffer PV(n) reads, right behind it.
      ok = ok && issue_s(par);
      for (int n = par; ok && n < nt; n += 2) {
        ok = issue_pv(n) && (n + 2 >= nt || issue_s(n + 2));
      }
      if (ok) umma_commit(bar(B_ALLDONE));
    } else if (lane == 0 && nt > 0) {
      umma_commit(bar(B_ALLDONE));  // a second issuer with no tile (nt == 1) still signs off
    }
  } else {
    // ---------------------------------------------------------------- softmax warps 0-7
    const int quarter = warp & 3;
    const int hf = warp >> 2;           // column half of S (keys) = index of this warp's O
    const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
    const int i = qt * 128 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t my_o = tmem + lane_off + kColO + 128 * hf;
    RowIntervals<MAXNI> ri;
    load_row_intervals(p.itab, b, p.NI, p.S, i, ri);
    bool ok = nt > 0;
    float m_run = -INFINITY;  // this half's running max (log2 domain)
    float l_run = 0.f;        // this half's running row sum
    const float sl2 = p.scale_log2;
    int kt = next_tile(bmrow, p.NT, 0);
    for (int n = 0; ok && n < nt; ++n, kt = next_tile(bmrow, p.NT, kt + 1)) {
      const int sb = n & 1;
      const bool s_ready = wait(bar(B_SFULL + sb), (n >> 1) & 1, 0x107);
      __syncwarp();
      if (!s_ready) { ok = false; break; }
      tc_fence_after();
      const uint32_t my_s = tmem + lane_off + kColS + sb * 128 + 64 * hf;
      float s[64];
      {
        uint32_t t0[32], t1[32];
        tmem_ld32(my_s, t0);
        tmem_ld32(my_s + 32, t1);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(t0[c]);
          s[32 + c] = __uint_as_float(t1[c]);
        }
      }
      if (!tile_is_full(bmrow, kt)) {
        const int j0 = kt * 128 + 64 * hf;
        mask_cols_any(s, j0, ri, p.NI, p.check, p.masked != 0);
      }
      // row max of the 64 scores as a tree of 3-input maxima (depth 4: 64 -> 22 -> 8 -> 3 -> 1),
      // so the two softmax warps of an SMSP do not wait on one long dependent chain
      float a[22], c8[8];
#pragma unroll
      for (int k = 0; k < 21; ++k) a[k] = max3f(s[3 * k], s[3 * k + 1], s[3 * k + 2]);
      a[21] = s[63];
#pragma unroll
      for (int k = 0; k < 7; ++k) c8[k] = max3f(a[3 * k], a[3 * k + 1], a[3 * k + 2]);
      c8[7] = a[21];
      const float m_tile =
          max3f(max3f(c8[0], c8[1], c8[2]), max3f(c8[3], c8[4], c8[5]), fmaxf(c8[6], c8[7])) * sl2;
      float alpha = 1.f;
      if (m_tile > m_run + 8.f) {  // also true when m_run = -inf and the tile has a visible key
        alpha = ex2_approx(m_run - m_tile);  // 0 when m_run = -inf
        m_run = m_tile;
      }
      const float moff = (m_run == -INFINITY) ? 0.f : m_run;
      // p = exp2(s * scale * log2e - m), two scores per paired FMA; row sums in paired adds
      const float2 scale2 = make_float2(sl2, sl2), neg_m2 = make_float2(-moff, -moff);
      float2 lsa = make_float2(0.f, 0.f), lsb = make_float2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float2 xa = fma2(make_float2(s[c], s[c + 1]), scale2, neg_m2);
        const float2 xb = fma2(make_float2(s[c + 2], s[c + 3]), scale2, neg_m2);
        const float2 pa = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
        const float2 pb = make_float2(ex2_approx(xb.x), ex2_approx(xb.y));
        lsa = add2(lsa, pa);
        lsb = add2(lsb, pb);
        pk[c / 2] = pack_bf16x2(pa.x, pa.y);
        pk[c / 2 + 1] = pack_bf16x2(pb.x, pb.y);
      }
      l_run = l_run * alpha + ((lsa.x + lsa.y) + (lsb.x + lsb.y));

      if (n >= 1 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        // rescale this half's O: PV(n-1) must be complete (PV(n-2) and earlier are, since S(n)
        // is).  Its stage barrier is at most one phase ahead of this wait: PV(n+2) needs this
        // warp's P(n+2).
        const bool o_ready = wait(bar(B_KVEMPTY + (n - 1) % kStages), ((n - 1) / kStages) & 1, 0x108);
        __syncwarp();
        if (!o_ready) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(my_o + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
          tmem_st32(my_o + c, o);
        }
      }
      // P over the S columns this warp has read: keys [64*hf, +64) -> columns [64*hf, +32)
      tmem_st32(my_s, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + sb));
    }

    // ---- epilogue: merge the two halves, O -> bf16, LSE (natural log) ----
    bool o_final = ok && wait(bar(B_ALLDONE), 0, 0x109);
    __syncwarp();
    // exchange (max, sum) with the warp of the other half through the Q tile, which no MMA
    // reads any more
    float m_other = -INFINITY, l_other = 0.f;
    if (o_final) {
      float2* slot = reinterpret_cast<float2*>(smem + L::kQ);  // [2 halves][128 rows]
      slot[hf * 128 + r] = make_float2(m_run, l_run);
      __syncwarp();
      const uint32_t pb = bar(B_PAIR + quarter);
      if (lane == 0) mbar_arrive(pb);
      o_final = wait(pb, 0, 0x10b);
      __syncwarp();
      if (o_final) {
        const float2 ot = slot[(hf ^ 1) * 128 + r];
        m_other = ot.x;
        l_other = ot.y;
      }
    }
    const float M = fmaxf(m_run, m_other);
    const float a_self = m_run == -INFINITY ? 0.f : ex2_approx(m_run - M);
    const float a_other = m_other == -INFINITY ? 0.f : ex2_approx(m_other - M);
    const float l_tot = l_run * a_self + l_other * a_other;
    __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.S + i) * D + hf * kHalf;
    if (o_final) {
      tc_fence_after();
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const float w0 = (hf == 0 ? a_self : a_other) * inv_l;  // weight of O_0
      const float w1 = (hf == 0 ? a_other : a_self) * inv_l;  // weight of O_1
#pragma unroll
      for (int c = 0; c < kHalf; c += 32) {
        uint32_t o0[32], o1[32];
        tmem_ld32(tmem + lane_off + kColO + hf * kHalf + c, o0);
        tmem_ld32(tmem + lane_off + kColO + 128 + hf * kHalf + c, o1);
        tmem_wait_ld();
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            y[e] = __uint_as_float(o0[8 * q + e]) * w0 + __uint_as_float(o1[8 * q + e]) * w1;
          uint4 v;
          v.x = pack_bf16x2(y[0], y[1]);
          v.y = pack_bf16x2(y[2], y[3]);
          v.z = pack_bf16x2(y[4], y[5]);
          v.w = pack_bf16x2(y[6], y[7]);
          dst[q] = v;
        }
      }
    } else {
      uint4* dst = reinterpret_cast<uint4*>(orow);
      for (int q = 0; q < kHalf / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
    }
    if (hf == 0)
      p.lse[static_cast<size_t>(bh) * p.S + i] =
          (o_final && l_tot > 0.f) ? (M + __log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up.  Copies and MMAs already issued still land in shared memory and TMEM:
    // wait for them before TMEM is freed and the CTA exits.
    if (warp == kProducerWarp && lane == 0 && nt > 0) {
      mbar_wait_drain(bar(B_Q), 0, p.status, 0x1f0);
      for (int s = 0; s < kStages && s < n_armed; ++s)
        mbar_wait_drain(bar(B_KVFULL + s), ((n_armed - 1 - s) / kStages) & 1, p.status, 0x1f1);
    }
    if ((warp == kMmaWarp || warp == kMmaWarp + 1) && lane == 0 && mma_issued) {
      umma_commit(bar(B_DRAIN + warp - kMmaWarp));
      mbar_wait_drain(bar(B_DRAIN + warp - kMmaWarp), 0, p.status, 0x1f2);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace fwd

template <int D, int MAXNI>
int fwd_launch(dim3 grid, cudaStream_t stream, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const FwdParams& p) {
  const uint32_t smem = fwd::Smem<D>::kAlloc;
  if (cudaFuncSetAttribute(fwd::attn_fwd_kernel<D, MAXNI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -1;
  fwd::attn_fwd_kernel<D, MAXNI><<<grid, fwd::kThreads, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_attn_fwd(const FwdParams& p, int d, const void* q, const void* k, const void* v,
                    cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const uint64_t rows = static_cast<uint64_t>(p.B) * p.H * p.S;
  if (!make_bf16_tile_map(&mq, q, rows, d) || !make_bf16_tile_map(&mk, k, rows, d) ||
      !make_bf16_tile_map(&mv, v, rows, d))
    return -1;
  const dim3 grid(p.B * p.NT * p.H);
  // interval registers: 4 cover every visible-form workload here; 9 the largest tables
  if (d == 128) {
    if (p.NI <= 4) return fwd_launch<128, 4>(grid, stream, mq, mk, mv, p);
    return fwd_launch<128, 9>(grid, stream, mq, mk, mv, p);
  }
  if (p.NI <= 4) return fwd_launch<64, 4>(grid, stream, mq, mk, mv, p);
  return fwd_launch<64, 9>(grid, stream, mq, mk, mv, p);
}

}  // namespace cm

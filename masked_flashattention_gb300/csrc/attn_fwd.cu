// Descriptor-guided attention, forward (CompileMask section 3.3.2), for sm_103a.
//
// One CTA computes one 128-row query tile of one (sample, head).  The Tile-State Bitmap row of
// that query tile lists the key tiles to visit: empty tiles are skipped, full tiles run without
// any mask, and partial tiles check every score against the row's intervals (mask.cuh), replacing
// invisible scores with -inf before the online softmax.
//
// Q stays in TMEM for the whole CTA: the softmax warps read their rows from global memory once
// and store them as bf16 pairs into TMEM, and S = Q K^T takes its A operand from there.  So the
// S MMAs read only K from shared memory (4 KB per 128x128x16 step instead of 8 KB), which keeps
// the tensor core's shared-memory reads well below the shared-memory bandwidth while TMA writes
// the next K and V tiles.
//
// Warp roles (320 threads):
//   warps 0-7  softmax.  Warp w serves TMEM lane quarter w % 4 (query rows 32*(w%4) ..) and
//              column half w / 4: keys [64*(w/4), +64) of each S tile and output columns
//              [(w/4)*d/2, +d/2) of O.  Per tile it reads its 64 scores from TMEM, masks partial
//              tiles, exchanges its local row maximum with the warp of the other key half (the
//              two share one running maximum, so one O accumulator serves both halves), writes P
//              (bf16 pairs) back over the S columns it has read, rescales its O columns when the
//              running maximum moved, and at the end writes its O columns and the LSE.
//   warp 8     TMA producer: K and V of each visited key tile into one of 3 stages (one barrier
//              for both tiles; the stage frees when the tile's PV MMAs completed).
//   warp 9     MMA issuer (one thread): S = Q K^T (Q from TMEM, K from shared memory) and
//              O += P V (P from TMEM, V from shared memory).
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256+d), Q [384, 384+d/2).  P of tile n
// lives in S buffer n % 2: keys [0,64) in columns [0,32), keys [64,128) in [64,96).
// Ordering without extra barriers: the MMA issues S(n+2) into a buffer only after it saw P(n) and
// issued PV(n), which reads P(n) from that buffer; tcgen05 MMAs of one thread run in issue order.
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
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kStages = 3;  // K ring and V ring depth

constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kColQ = 384;

template <int D>
struct Smem {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kKV = 0;  // stage s: K at kKV + 2*s*tile, V right after it
  // per-tile row-maximum exchange [2 slots][2 halves][128 rows], then the final row-sum exchange
  // [2 halves][128 rows]
  static constexpr uint32_t kXchg = kKV + kStages * 2u * kTileBytes;
  static constexpr uint32_t kBar = kXchg + 3u * 1024u;
  static constexpr uint32_t kRow = kBar + 256u;  // bitmap row: at most 64 words (NT <= 1024)
  static constexpr uint32_t kTotal = kRow + 256u;
  static constexpr uint32_t kAlloc = kTotal + 1024u;  // slack for 1024-byte alignment
};
static_assert(Smem<128>::kAlloc <= 232448, "forward shared memory exceeds 227 KB");

// The MMA thread waits twice per key tile (P ready, next K/V landed) and commits twice (S ready,
// PV done): every wait of the issuing thread leaves a gap in the tensor pipe, so the barriers are
// shared where the ordering allows it.
enum {
  B_QT = 0,       // Q stored in TMEM by the softmax warps (8 arrivals)
  B_KVFULL = 1,   // +stage: K and V of a key tile landed (TMA, 2 tiles of bytes)
  B_KVEMPTY = 4,  // +stage: S and PV of the stage's tile have completed (also "O is up to date")
  B_SFULL = 7,    // +buffer
  B_PFULL = 9,    // +buffer: P of a tile in that S buffer, both halves (8 arrivals)
  B_XCHG = 11,    // +2*quarter+slot: row-maximum exchange of a warp pair (2 arrivals)
  B_PAIR = 19,    // +quarter: final row-sum exchange of a warp pair (2 arrivals, once)
  B_ALLDONE = 23, // every MMA of the CTA has completed (once)
  B_DRAIN = 24,   // abort path only: every MMA issued so far has completed
  B_COUNT = 25
};

template <int D, int MAXNI>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ FwdParams p) {
  using L = Smem<D>;
  constexpr int kHalf = D / 2;  // output columns of a softmax warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * B_COUNT + 4);
  int* s_ntiles = reinterpret_cast<int*>(smem + L::kBar + 8 * B_COUNT + 8);
  uint32_t* bmrow = reinterpret_cast<uint32_t*>(smem + L::kRow);
  float* xmax = reinterpret_cast<float*>(smem + L::kXchg);          // [2][2][128]
  float* xsum = reinterpret_cast<float*>(smem + L::kXchg + 2048u);  // [2][128]
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
    mbar_init(bar(B_QT), kSoftmaxWarps);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KVFULL + s), 1);
      mbar_init(bar(B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), kSoftmaxWarps);
    }
    for (int s = 0; s < 8; ++s) mbar_init(bar(B_XCHG + s), 2);
    for (int s = 0; s < 4; ++s) mbar_init(bar(B_PAIR + s), 2);
    mbar_init(bar(B_ALLDONE), 1);
    mbar_init(bar(B_DRAIN), 1);
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
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int row0 = bh * p.S;
      int kt = next_tile(bmrow, p.NT, 0);
      for (int n = 0; n < nt; ++n, kt = next_tile(bmrow, p.NT, kt + 1)) {
        const int st = n % kStages;
        if (n >= kStages && !wait(bar(B_KVEMPTY + st), ((n / kStages) - 1) & 1, 0x101)) break;
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
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idS = make_idesc_bf16(128, 128, 0, 0);  // A = Q (TMEM), B = K K-major
      constexpr uint32_t idO = make_idesc_bf16(128, D, 0, 1);    // A = P (TMEM), B = V MN-major
      bool ok = wait(bar(B_QT), 0, 0x102);
      // O += P V for tile m: P keys [0,64) at S columns [0,32), keys [64,128) at [64,96).  V(m)
      // landed before S(m) was issued (same barrier as K(m)).
      auto issue_pv = [&](int m) -> bool {
        const int st = m % kStages;
        // one barrier per S buffer: the softmax warps can be at most one tile ahead of this
        // wait, so a barrier never runs two phases ahead of its waiter
        if (!wait(bar(B_PFULL + (m & 1)), (m >> 1) & 1, 0x103)) return false;
        tc_fence_after();
        const uint32_t dV = sdesc_lo(sbase + L::kKV + st * 2u * L::kTileBytes + L::kTileBytes, 16384u);
        const uint32_t sP = tmem + kColS + (m & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_lo(tmem + kColO, sP + 64 * (kk >> 2) + 8 * (kk & 3), dV + kstep_mnmajor(kk), idO,
                     (m > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(B_KVEMPTY + st));
        return true;
      };
      // S(n) into buffer n % 2 = Q K(n)^T, Q from TMEM
      auto issue_s = [&](int n) -> bool {
        const int st = n % kStages;
        if (!wait(bar(B_KVFULL + st), (n / kStages) & 1, 0x105)) return false;
        tc_fence_after();
        mma_issued = true;
        const uint32_t dK = sdesc_lo(sbase + L::kKV + st * 2u * L::kTileBytes, 16u);
        const uint32_t dS = tmem + kColS + (n & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ts_lo(dS, tmem + kColQ + 8 * kk, dK + kstep_kmajor(kk), idS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL + (n & 1)));
        return true;
      };
      // Both S buffers first; then per tile: PV(n) as soon as its P is written, and S(n+2) into
      // the buffer PV(n) reads, right behind it.  The thread waits for P with nothing queued
      // behind the wait, so it issues PV the moment P arrives.
      if (ok) tc_fence_after();
      ok = ok && issue_s(0) && (nt < 2 || issue_s(1));
      for (int n = 0; ok && n < nt; ++n) {
        ok = issue_pv(n) && (n + 2 >= nt || issue_s(n + 2));
      }
      if (ok) umma_commit(bar(B_ALLDONE));
    }
  } else {
    // ---------------------------------------------------------------- softmax warps 0-7
    const int quarter = warp & 3;
    const int hf = warp >> 2;           // key half of S, and output-column half of O
    const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
    const int i = qt * 128 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t my_o = tmem + lane_off + kColO + hf * kHalf;
    // Q row i, this warp's half of its bf16 pairs, into the Q columns of TMEM
    if (nt > 0) {
      const uint4* qrow = reinterpret_cast<const uint4*>(
          p.q + (static_cast<size_t>(bh) * p.S + i) * D + hf * kHalf);
      if constexpr (D == 128) {
        uint32_t w[32];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const uint4 v = qrow[x];
          w[4 * x] = v.x;
          w[4 * x + 1] = v.y;
          w[4 * x + 2] = v.z;
          w[4 * x + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + kColQ + hf * 32, w);
      } else {
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint4 v = qrow[x];
          w[4 * x] = v.x;
          w[4 * x + 1] = v.y;
          w[4 * x + 2] = v.z;
          w[4 * x + 3] = v.w;
        }
        tmem_st16(tmem + lane_off + kColQ + hf * 16, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QT));
    }
    RowIntervals<MAXNI> ri;
    load_row_intervals(p.itab, b, p.NI, p.S, i, ri);
    bool ok = nt > 0;
    float m_run = -INFINITY;  // the row's running max (log2 domain), shared by the warp pair
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
      // row max of the 64 scores as a tree of 3-input maxima (depth 4: 64 -> 22 -> 8 -> 3 -> 1)
      float a[22], c8[8];
#pragma unroll
      for (int k = 0; k < 21; ++k) a[k] = max3f(s[3 * k], s[3 * k + 1], s[3 * k + 2]);
      a[21] = s[63];
#pragma unroll
      for (int k = 0; k < 7; ++k) c8[k] = max3f(a[3 * k], a[3 * k + 1], a[3 * k + 2]);
      c8[7] = a[21];
      const float m_loc =
          max3f(max3f(c8[0], c8[1], c8[2]), max3f(c8[3], c8[4], c8[5]), fmaxf(c8[6], c8[7])) * sl2;
      // the tile's row max over both key halves: exchange with the warp of the other half
      const int slot = n & 1;
      xmax[(slot * 2 + hf) * 128 + r] = m_loc;
      __syncwarp();
      const uint32_t xb = bar(B_XCHG + 2 * quarter + slot);
      if (lane == 0) mbar_arrive(xb);
      const bool x_ready = wait(xb, (n >> 1) & 1, 0x10a);
      __syncwarp();
      if (!x_ready) { ok = false; break; }
      const float m_tile = fmaxf(m_loc, xmax[(slot * 2 + (hf ^ 1)) * 128 + r]);
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
        const float2 xb2 = fma2(make_float2(s[c + 2], s[c + 3]), scale2, neg_m2);
        const float2 pa = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
        const float2 pb = make_float2(ex2_approx(xb2.x), ex2_approx(xb2.y));
        lsa = add2(lsa, pa);
        lsb = add2(lsb, pb);
        pk[c / 2] = pack_bf16x2(pa.x, pa.y);
        pk[c / 2 + 1] = pack_bf16x2(pb.x, pb.y);
      }
      l_run = l_run * alpha + ((lsa.x + lsa.y) + (lsb.x + lsb.y));

      if (n >= 1 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        // rescale this warp's O columns: PV(n-1) must be complete (PV(n-2) and earlier are,
        // since S(n) is).  Its stage barrier is at most one phase ahead of this wait: PV(n+2)
        // needs this warp's P(n+2).
        const bool o_ready = wait(bar(B_KVEMPTY + (n - 1) % kStages), ((n - 1) / kStages) & 1, 0x108);
        __syncwarp();
        if (!o_ready) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kHalf; c += 32) {
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

    // ---- epilogue: row sum over both halves, O -> bf16, LSE (natural log) ----
    bool o_final = ok && wait(bar(B_ALLDONE), 0, 0x109);
    __syncwarp();
    float l_other = 0.f;
    if (o_final) {
      xsum[hf * 128 + r] = l_run;
      __syncwarp();
      const uint32_t pb = bar(B_PAIR + quarter);
      if (lane == 0) mbar_arrive(pb);
      o_final = wait(pb, 0, 0x10b);
      __syncwarp();
      if (o_final) l_other = xsum[(hf ^ 1) * 128 + r];
    }
    const float l_tot = l_run + l_other;
    __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.S + i) * D + hf * kHalf;
    if (o_final) {
      tc_fence_after();
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll
      for (int c = 0; c < kHalf; c += 32) {
        uint32_t o[32];
        tmem_ld32(my_o + c, o);
        tmem_wait_ld();
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
          v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
          v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
          v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
          dst[q] = v;
        }
      }
    } else {
      uint4* dst = reinterpret_cast<uint4*>(orow);
      for (int q = 0; q < kHalf / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
    }
    if (hf == 0)
      p.lse[static_cast<size_t>(bh) * p.S + i] =
          (o_final && l_tot > 0.f) ? (m_run + __log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up.  Copies and MMAs already issued still land in shared memory and TMEM:
    // wait for them before TMEM is freed and the CTA exits.
    if (warp == kProducerWarp && lane == 0 && nt > 0) {
      for (int s = 0; s < kStages && s < n_armed; ++s)
        mbar_wait_drain(bar(B_KVFULL + s), ((n_armed - 1 - s) / kStages) & 1, p.status, 0x1f1);
    }
    if (warp == kMmaWarp && lane == 0 && mma_issued) {
      umma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, p.status, 0x1f2);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace fwd

template <int D, int MAXNI>
int fwd_launch(dim3 grid, cudaStream_t stream, const CUtensorMap& mk, const CUtensorMap& mv,
               const FwdParams& p) {
  const uint32_t smem = fwd::Smem<D>::kAlloc;
  if (cudaFuncSetAttribute(fwd::attn_fwd_kernel<D, MAXNI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -1;
  fwd::attn_fwd_kernel<D, MAXNI><<<grid, fwd::kThreads, smem, stream>>>(mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_attn_fwd(const FwdParams& p, int d, const void* k, const void* v, cudaStream_t stream) {
  CUtensorMap mk, mv;
  const uint64_t rows = static_cast<uint64_t>(p.B) * p.H * p.S;
  if (!make_bf16_tile_map(&mk, k, rows, d) || !make_bf16_tile_map(&mv, v, rows, d)) return -1;
  const dim3 grid(p.B * p.NT * p.H);
  // interval registers: 4 cover every visible-form workload here; 9 the largest tables
  if (d == 128) {
    if (p.NI <= 4) return fwd_launch<128, 4>(grid, stream, mk, mv, p);
    return fwd_launch<128, 9>(grid, stream, mk, mv, p);
  }
  if (p.NI <= 4) return fwd_launch<64, 4>(grid, stream, mk, mv, p);
  return fwd_launch<64, 9>(grid, stream, mk, mv, p);
}

}  // namespace cm

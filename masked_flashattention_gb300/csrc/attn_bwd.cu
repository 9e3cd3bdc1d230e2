// Descriptor-guided attention, backward, dK and dV (CompileMask sections 3.2.2 / 3.3 / 3.3.2),
// for sm_103a.
//
// The backward pass traverses key tiles, so it uses the backward descriptor: per key column j,
// the visible query intervals, and per (key tile, query tile) the 2-bit state.  One CTA owns one
// 128-key tile of one (sample, head) and walks the non-empty query tiles of its bitmap row:
//
//   S^T  = K Q^T            (tcgen05, TMEM)        P^T  = exp2(S^T * scale*log2e - LSE*log2e)
//   dP^T = V dO^T           (tcgen05, TMEM)        dS^T = P^T * (dP^T - D),  D = rowsum(dO * O)
//   dK  += dS^T Q           (TMEM accumulator; dS^T is the A operand, read from TMEM)
//   dV  += P^T dO           (TMEM accumulator; P^T is the A operand, read from TMEM)
//
// dQ is computed by a second kernel that walks query tiles (attn_dq.cu); adding every key tile's
// dQ partial into an fp32 accumulator here would make L2 read-modify-write traffic the bound.
//
// Partial tiles check each query index against the key column's intervals with the unsigned
// test of section 4.4 and zero P there (the -inf of the forward); full tiles skip the check.
// Empty tiles are never visited.
//
// Warp roles (320 threads):
//   warps 0-7  compute.  Warp w serves TMEM lane quarter w % 4 (key rows 32*(w%4) ..) and column
//              half w / 4: queries [64*half, +64) of S^T / dP^T and head-dim columns
//              [half*d/2, +d/2) of dV and dK.
//   warp 8     TMA producer: K, V once; per query tile Q and dO (+ LSE*log2e and D by bulk
//              copy) into one of two slots, one barrier per slot.
//   warp 9     MMA issuer (one thread).
// TMEM (512 columns): dV [0, d), dK [128, 128+d), and two 128-column regions RA [256, 384),
// RB [384, 512) whose roles alternate between query tiles.  For tile m with X = RA (m even) or
// RB (m odd) and Y the other one:
//   S^T(m) -> X; the compute warps overwrite it in place with the bf16 P^T pairs (each warp
//   writes only columns it has already read); dP^T(m) -> Y.
//   The compute warps then write the bf16 dS^T pairs into the other half of the columns they read
//   from X (warp half h: P^T at 64h + [0,32), dS^T at 64h + [32,64)).
//   As soon as P^T is written the MMA issues dV(m) (A = P^T from X) while the compute warps form
//   dS^T; once dS^T is written it issues S^T(m+1) -> Y (its dP^T was consumed), dK(m) (A = dS^T
//   from X) and dP^T(m+1) -> X (after dV and dK read it).  Both gradient MMAs take their A operand
//   from TMEM, so shared memory carries only K, V, Q and dO, and the next tile's P overlaps dK.
// Shared memory: K, V, Q and dO (two slots each, 128-byte swizzle), LSE*log2e and D (per slot),
// barriers, and the CTA's row of the backward bitmap (the non-empty query tiles are found by
// scanning it).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "kernels.h"
#include "mask.cuh"
#include "ptx.cuh"
#include "tma_host.h"

namespace cm {

namespace bwd {

constexpr int kComputeWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;

constexpr uint32_t kColDV = 0;
constexpr uint32_t kColDK = 128;
constexpr uint32_t kColRA = 256;
constexpr uint32_t kColRB = 384;

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Smem {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kTileBytes;
  static constexpr uint32_t kQ = 2 * kTileBytes;      // two slots
  static constexpr uint32_t kdO = 4 * kTileBytes;      // two slots
  static constexpr uint32_t kLse2 = 6 * kTileBytes;    // [2 slots][128 floats]: -LSE * log2(e)
  static constexpr uint32_t kDelta = kLse2 + 1024u;    // [2 slots][128 floats]: -D
  static constexpr uint32_t kBar = kDelta + 1024u;
  static constexpr uint32_t kRow = kBar + 256u;        // bitmap row: at most 64 words (NT <= 1024)
  static constexpr uint32_t kTotal = kRow + 256u;
  static constexpr uint32_t kAlloc = kTotal + 1024u;  // + slack to align the base to 1024 bytes
};
static_assert(Smem<128>::kAlloc <= 232448, "backward shared memory exceeds 227 KB");

enum {
  B_KV = 0,        // K and V loaded
  B_QFULL = 1,     // +slot: Q, dO, LSE*log2e and D of a query tile loaded (one barrier: each
                   // wait of the MMA thread leaves a gap in the tensor pipe)
  B_QEMPTY = 3,    // +slot: the dK MMA (last reader of the slot, after dV) is done
  B_SFULL = 5,     // S^T of the current tile computed
  B_DPFULL = 6,    // dP^T of the current tile computed
  B_PDS = 7,       // compute warps wrote dS^T (TMEM) and read dP^T (8 arrivals)
  B_DONE = 8,      // every MMA of the CTA completed (dK, dV final)
  B_PREADY = 9,    // compute warps wrote P^T (TMEM) (8 arrivals)
  B_DRAIN = 10,    // abort path only: every MMA issued so far has completed
  B_COUNT = 11
};


__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// P^T of 32 queries of this key row: p = exp2(s * scale*log2e + (-LSE*log2e)) in fp32 (kept for
// dS) and as bf16 pairs (the A operand of dV).  Shared memory holds -LSE*log2e per query, so the
// exponent is one paired FMA.  For a partial tile, queries whose bit in `vis` is clear get p = 0.
template <bool FULL>
__device__ __forceinline__ void p_chunk(const uint32_t (&sr)[32], uint32_t lse2_addr, float sl2,
                                        uint32_t vis, float (&pf)[32], uint32_t (&pp)[16]) {
  const float2 scale2 = make_float2(sl2, sl2);
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const float4 l4 = ld_shared_f4(lse2_addr + c * 4u);
    const float2 xa = fma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), scale2,
                           make_float2(l4.x, l4.y));
    const float2 xb = fma2(make_float2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])),
                           scale2, make_float2(l4.z, l4.w));
    pf[c] = ex2_approx(xa.x);
    pf[c + 1] = ex2_approx(xa.y);
    pf[c + 2] = ex2_approx(xb.x);
    pf[c + 3] = ex2_approx(xb.y);
    if (!FULL) {
#pragma unroll
      for (int e = 0; e < 4; ++e) pf[c + e] = ((vis >> (c + e)) & 1u) ? pf[c + e] : 0.f;
    }
    pp[c / 2] = pack_bf16x2(pf[c], pf[c + 1]);
    pp[c / 2 + 1] = pack_bf16x2(pf[c + 2], pf[c + 3]);
  }
}

// dS^T of 32 queries: ds = p * (dp + (-D)), as bf16 pairs.
__device__ __forceinline__ void ds_chunk(const float (&pf)[32], const uint32_t (&dpr)[32],
                                         uint32_t delta_addr, uint32_t (&dd)[16]) {
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const float4 d4 = ld_shared_f4(delta_addr + c * 4u);
    const float2 ga = add2(make_float2(__uint_as_float(dpr[c]), __uint_as_float(dpr[c + 1])),
                           make_float2(d4.x, d4.y));
    const float2 gb = add2(make_float2(__uint_as_float(dpr[c + 2]), __uint_as_float(dpr[c + 3])),
                           make_float2(d4.z, d4.w));
    const float2 dsa = mul2(make_float2(pf[c], pf[c + 1]), ga);
    const float2 dsb = mul2(make_float2(pf[c + 2], pf[c + 3]), gb);
    dd[c / 2] = pack_bf16x2(dsa.x, dsa.y);
    dd[c / 2 + 1] = pack_bf16x2(dsb.x, dsb.y);
  }
}

template <int D, int MAXNI>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ BwdParams p) {
  using L = Smem<D>;
  constexpr int kHalf = D / 2;           // head-dim columns per compute warp
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
  const int kt = item & 0xFFFF;
  if (b < 0 || b >= p.B || kt >= p.NT) {  // a schedule entry that no descriptor build wrote
    if (threadIdx.x == 0) set_status(p.status, kDevBadSchedule, item_idx);
    return;
  }
  const int bh = b * p.H + h;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_KV), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(B_QFULL + x), 1);
      mbar_init(bar(B_QEMPTY + x), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_DPFULL), 1);
    mbar_init(bar(B_PDS), kComputeWarps);
    mbar_init(bar(B_DONE), 1);
    mbar_init(bar(B_PREADY), kComputeWarps);
    mbar_init(bar(B_DRAIN), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    // this CTA's bitmap row (W <= 64 words) and its count of non-empty query tiles
    const uint32_t* row = p.bm + (static_cast<size_t>(b) * p.NT + kt) * p.W;
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
  const int row0 = bh * p.S;
  // asynchronous work issued so far, for the abort path: query-tile slots armed (producer), any
  // MMA issued (MMA thread)
  int m_armed = 0;
  bool mma_issued = false;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar(B_KV), 2 * L::kTileBytes);
      for (int x = 0; x < D / 64; ++x) {
        tma_load_2d(sbase + L::kK + x * 16384u, &tmK, x * 64, row0 + kt * 128, bar(B_KV));
        tma_load_2d(sbase + L::kV + x * 16384u, &tmV, x * 64, row0 + kt * 128, bar(B_KV));
      }
      int qt = next_tile(bmrow, p.NT, 0);
      for (int m = 0; m < nt; ++m, qt = next_tile(bmrow, p.NT, qt + 1)) {
        const int slot = m & 1;
        const size_t r = static_cast<size_t>(row0) + qt * 128;
        // a slot is free once the dK MMA of the tile two back (its last reader) is done
        if (m >= 2 && !wait(bar(B_QEMPTY + slot), ((m - 2) >> 1) & 1, 0x201))
          break;
        const uint32_t full = bar(B_QFULL + slot);
        m_armed = m + 1;
        mbar_arrive_expect_tx(full, 2u * (L::kTileBytes + 512u));
        for (int x = 0; x < D / 64; ++x) {
          tma_load_2d(sbase + L::kQ + slot * L::kTileBytes + x * 16384u, &tmQ, x * 64,
                      row0 + qt * 128, full);
          tma_load_2d(sbase + L::kdO + slot * L::kTileBytes + x * 16384u, &tmdO, x * 64,
                      row0 + qt * 128, full);
        }
        bulk_load(sbase + L::kLse2 + slot * 512u, p.lse2 + r, 512u, full);
        bulk_load(sbase + L::kDelta + slot * 512u, p.delta + r, 512u, full);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idSS = make_idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
      constexpr uint32_t idKM = make_idesc_bf16(128, D, 0, 1);    // dK, dV
      const uint32_t sK = sbase + L::kK, sV = sbase + L::kV;
      // low words of the shared-memory descriptors (the split form keeps the issue loop short:
      // the issuing thread shares its SM sub-partition with two compute warps, and every
      // instruction it needs between MMAs leaves the tensor pipe waiting longer)
      const uint32_t dK0 = sdesc_lo(sK, 16u), dV0 = sdesc_lo(sV, 16u);
      const uint32_t dQ0 = sdesc_lo(sbase + L::kQ, 16u), ddO0 = sdesc_lo(sbase + L::kdO, 16u);
      // tile 0: S^T -> RA, dP^T -> RB
      bool ok = wait(bar(B_KV), 0, 0x202) &&
                wait(bar(B_QFULL), 0, 0x203);
      if (ok) {
        tc_fence_after();
        mma_issued = true;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_lo(tmem + kColRA, dK0 + kstep_kmajor(kk), dQ0 + kstep_kmajor(kk), idSS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL));
      }
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_lo(tmem + kColRB, dV0 + kstep_kmajor(kk), ddO0 + kstep_kmajor(kk), idSS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_DPFULL));
      }
      for (int m = 0; ok && m < nt; ++m) {
        const uint32_t X = (m & 1) ? kColRB : kColRA;
        const uint32_t Y = (m & 1) ? kColRA : kColRB;
        const uint32_t sQ = sbase + L::kQ + (m & 1) * L::kTileBytes;
        const uint32_t sdO = sbase + L::kdO + (m & 1) * L::kTileBytes;
        // dV += P^T dO as soon as P^T is in X, while the compute warps work on dS^T.
        // P^T pairs: queries [0,64) at X columns [0,32), [64,128) at [64,96)
        if (!wait(bar(B_PREADY), m & 1, 0x210)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_lo(tmem + kColDV, tmem + X + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                     sdesc_lo(sdO, 16384u) + kstep_mnmajor(kk), idKM, (m > 0 || kk > 0) ? 1u : 0u);
        if (!wait(bar(B_PDS), m & 1, 0x205)) break;
        tc_fence_after();
        if (m + 1 < nt) {
          // the next tile's S^T into Y (its dP^T was consumed), so that its P can start while
          // the tensor pipe runs dK
          const uint32_t sQn = sbase + L::kQ + ((m + 1) & 1) * L::kTileBytes;
          if (!wait(bar(B_QFULL + ((m + 1) & 1)), ((m + 1) >> 1) & 1, 0x203))
            break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss_lo(tmem + Y, dK0 + kstep_kmajor(kk), sdesc_lo(sQn, 16u) + kstep_kmajor(kk), idSS,
                       kk > 0 ? 1u : 0u);
          umma_commit(bar(B_SFULL));
        }
        // dK += dS^T Q with dS^T read from X: queries [64h + 32c, +32) at columns 64h + 32 + 16c
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_lo(tmem + kColDK, tmem + X + 64 * (kk >> 2) + 32 + 8 * (kk & 3),
                     sdesc_lo(sQ, 16384u) + kstep_mnmajor(kk), idKM, (m > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(B_QEMPTY + (m & 1)));
        if (m + 1 < nt) {
          // dP^T of the next tile into X, after dV and dK above have read P^T and dS^T from it
          // (its dO landed with its Q, waited for before S^T)
          const uint32_t sdOn = sbase + L::kdO + ((m + 1) & 1) * L::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss_lo(tmem + X, dV0 + kstep_kmajor(kk), sdesc_lo(sdOn, 16u) + kstep_kmajor(kk), idSS,
                       kk > 0 ? 1u : 0u);
          umma_commit(bar(B_DPFULL));
        } else {
          umma_commit(bar(B_DONE));
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- compute warps 0-7
    const int quarter = warp & 3;
    const int hf = warp >> 2;
    const int r = quarter * 32 + lane;  // key row (S^T, dP^T, dV, dK)
    const int j = kt * 128 + r;         // key column owned for S^T / dP^T
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    if (warp == 0 && h == 0) {
      // The backward descriptor must describe the transposed mask of the forward one: tile
      // (kt, q) of this bitmap row has the state of tile (q, kt) of the forward bitmap.  Checked
      // once per key tile (head 0); a mismatch (two MaskSpecs that do not describe the same
      // mask) is recorded in the status word, the computation goes on.
      bool bad = false;
      for (int q = lane; q < p.NT; q += 32) {
        const uint32_t cb = (bmrow[q >> 4] >> (2 * (q & 15))) & 3u;
        const uint32_t cf =
            (p.bm_f[(static_cast<size_t>(b) * p.NT + q) * p.W + (kt >> 4)] >> (2 * (kt & 15))) & 3u;
        bad |= cb != cf;
      }
      if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_status(p.status, kDevDescMismatch, kt);
    }
    RowIntervals<MAXNI> ri;
    load_row_intervals(p.itab, b, p.NI, p.S, j, ri);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int qt = next_tile(bmrow, p.NT, 0);
    for (int m = 0; ok && m < nt; ++m, qt = next_tile(bmrow, p.NT, qt + 1)) {
      const bool full = tile_is_full(bmrow, qt);
      const uint32_t X = (m & 1) ? kColRB : kColRA;
      const uint32_t Y = (m & 1) ? kColRA : kColRB;

      // ---- P^T: S^T from X, written back in place as bf16 pairs; fp32 P kept for dS ----
      bool ready = wait(bar(B_SFULL), m & 1, 0x206) &&
                   wait(bar(B_QFULL + (m & 1)), (m >> 1) & 1, 0x207);
      __syncwarp();
      if (!ready) { ok = false; break; }
      tc_fence_after();
      float pf[2][32];
      const uint32_t lse2_base = sbase + L::kLse2 + (m & 1) * 512u;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int q0 = 64 * hf + 32 * ch;  // first query of the chunk within the tile
        uint32_t sr[32], pp[16];
        tmem_ld32(tmem + lane_off + X + q0, sr);
        tmem_wait_ld();
        if (full) {
          p_chunk<true>(sr, lse2_base + q0 * 4u, sl2, 0u, pf[ch], pp);
        } else {
          const int i0 = qt * 128 + q0;
          const uint32_t vis = visible_bits_any(i0, ri, p.NI, p.check, p.masked != 0);
          p_chunk<false>(sr, lse2_base + q0 * 4u, sl2, vis, pf[ch], pp);
        }
        // P^T pairs into X columns this warp has already read: hf * 64 + ch * 16
        tmem_st16(tmem + lane_off + X + hf * 64 + ch * 16, pp);
      }

      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PREADY));

      // ---- dS^T = P^T * (dP^T - D): dP^T from Y; dS^T as bf16 pairs into X ----
      ready = wait(bar(B_DPFULL), m & 1, 0x20e);
      __syncwarp();
      if (!ready) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int q0 = 64 * hf + 32 * ch;
        uint32_t dpr[32], dd[16];
        tmem_ld32(tmem + lane_off + Y + q0, dpr);
        tmem_wait_ld();
        ds_chunk(pf[ch], dpr, sbase + L::kDelta + (m & 1) * 512u + q0 * 4u, dd);
        // dS^T pairs into X columns this warp has read and P^T does not use: 64 hf + 32 + 16 ch
        tmem_st16(tmem + lane_off + X + hf * 64 + 32 + ch * 16, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PDS));

    }
    __syncwarp();

    // ---- epilogue: dV, dK (scaled) -> bf16, this warp's half of the head dim ----
    __nv_bfloat16* dvrow = p.dv + (static_cast<size_t>(row0) + j) * D + hf * kHalf;
    __nv_bfloat16* dkrow = p.dk + (static_cast<size_t>(row0) + j) * D + hf * kHalf;
    const bool done = nt > 0 && ok && wait(bar(B_DONE), 0, 0x20f);
    __syncwarp();
    if (done) {
      tc_fence_after();
      const float sc = p.scale;
      // dV, then dK (scaled), as bf16 pairs of this row's columns, stored a warp's 32 rows at a
      // time with coalesced stores
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        uint32_t ob[kHalf / 2];
#pragma unroll
        for (int c = 0; c < kHalf; c += 32) {
          uint32_t a[32];
          tmem_ld32(tmem + lane_off + (x == 0 ? kColDV : kColDK) + hf * kHalf + c, a);
          tmem_wait_ld();
          const float f = x == 0 ? 1.f : sc;
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            ob[(c + e) / 2] = pack_bf16x2(__uint_as_float(a[e]) * f, __uint_as_float(a[e + 1]) * f);
        }
        __nv_bfloat16* rowp = x == 0 ? dvrow : dkrow;
        store_rows_coalesced<kHalf / 8>(
            ob, reinterpret_cast<char*>(rowp - static_cast<size_t>(lane) * D), D * 2u, lane);
      }
    } else {
      uint4* dva = reinterpret_cast<uint4*>(dvrow);
      uint4* dka = reinterpret_cast<uint4*>(dkrow);
      for (int q = 0; q < kHalf / 8; ++q) {
        dva[q] = make_uint4(0, 0, 0, 0);
        dka[q] = make_uint4(0, 0, 0, 0);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up.  Copies and MMAs already issued still land in shared memory and TMEM:
    // wait for them before TMEM is freed and the CTA exits.
    if (warp == kProducerWarp && lane == 0 && nt > 0) {
      mbar_wait_drain(bar(B_KV), 0, p.status, 0x2f0);
      for (int s = 0; s < 2 && s < m_armed; ++s)
        mbar_wait_drain(bar(B_QFULL + s), ((m_armed - 1 - s) >> 1) & 1, p.status, 0x2f1);
    }
    if (warp == kMmaWarp && lane == 0 && mma_issued) {
      umma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, p.status, 0x2f2);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// Per row, negated for the paired FMAs of the backward kernels: -D = -sum_c dO[c] * O[c] (fp32)
// and -LSE * log2(e) (-inf for a row that sees nothing, so that its P is exp2(-inf) = 0).  One
// warp per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_prologue_kernel(const __nv_bfloat16* o,
                                                           const __nv_bfloat16* d_o,
                                                           const float* lse, float* delta,
                                                           float* lse2, size_t rows) {
  const size_t row = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr int kPer = D / 32;  // elements per lane (2 or 4)
  const __nv_bfloat16* a = o + row * D + lane * kPer;
  const __nv_bfloat16* g = d_o + row * D + lane * kPer;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc += __bfloat162float(a[e]) * __bfloat162float(g[e]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (lane == 0) {
    delta[row] = -acc;
    const float l = lse[row];
    lse2[row] = l == -INFINITY ? -INFINITY : -l * kLog2e;
  }
}

}  // namespace bwd

int launch_bwd_prologue(int d, const void* o, const void* d_o, const float* lse, float* delta,
                        float* lse2, size_t rows, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  if (d == 128)
    bwd::bwd_prologue_kernel<128><<<blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), lse, delta,
        lse2, rows);
  else
    bwd::bwd_prologue_kernel<64><<<blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), lse, delta,
        lse2, rows);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <int D, int MAXNI>
int bwd_launch(dim3 grid, cudaStream_t stream, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo, const BwdParams& p) {
  const uint32_t smem = bwd::Smem<D>::kAlloc;
  if (cudaFuncSetAttribute(bwd::attn_bwd_kernel<D, MAXNI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -1;
  bwd::attn_bwd_kernel<D, MAXNI><<<grid, bwd::kThreads, smem, stream>>>(mq, mk, mv, mdo, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_attn_dkdv(const BwdParams& p, int d, const void* q, const void* k, const void* v,
                     const void* d_o, cudaStream_t stream) {
  const size_t rows = static_cast<size_t>(p.B) * p.H * p.S;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_bf16_tile_map(&mq, q, rows, d) || !make_bf16_tile_map(&mk, k, rows, d) ||
      !make_bf16_tile_map(&mv, v, rows, d) || !make_bf16_tile_map(&mdo, d_o, rows, d))
    return -1;
  const dim3 grid(p.B * p.NT * p.H);
  // interval registers: 4 cover every visible-form workload here; 9 the largest tables
  if (d == 128) {
    if (p.NI <= 4) return bwd_launch<128, 4>(grid, stream, mq, mk, mv, mdo, p);
    return bwd_launch<128, 9>(grid, stream, mq, mk, mv, mdo, p);
  }
  if (p.NI <= 4) return bwd_launch<64, 4>(grid, stream, mq, mk, mv, mdo, p);
  return bwd_launch<64, 9>(grid, stream, mq, mk, mv, mdo, p);
}

}  // namespace cm

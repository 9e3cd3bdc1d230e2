// Descriptor-guided attention, backward, dK and dV (CompileMask sections 3.2.2 / 3.3 / 3.3.2),
// for sm_103a.
//
// The backward pass traverses key tiles, so it uses the backward descriptor: per key column j,
// the visible query intervals, and per (key tile, query tile) the 2-bit state.  A work item is one
// 128-key tile of one (sample, head); its CTA walks the non-empty query tiles of the item's
// bitmap row:
//
//   S^T  = K Q^T            (tcgen05, TMEM)        P^T  = exp2(S^T * scale*log2e - LSE*log2e)
//   dP^T = V dO^T           (tcgen05, TMEM)        dS^T = P^T * (dP^T - D),  D = rowsum(dO * O)
//   dK  += dS^T Q           (TMEM accumulator; dS^T is the A operand, read from TMEM)
//   dV  += P^T dO           (TMEM accumulator; P^T is the A operand, read from TMEM)
//
// The CTAs are persistent (one per SM).  The producer warp takes items from a work queue in the
// descriptor's status buffer (atomic counter over the schedule, longest bitmap rows first) and
// stages each item's bitmap row and description into one of two buffers, so the next item's K, V
// and first query tiles load while the current item's gradients are written.  LSE*log2e and -D
// per query row come from the workspace that the dQ kernel fills; this kernel runs after it.
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
//   warp 8     producer: work queue, bitmap row; TMA of K, V once per item; per query tile Q
//              and dO (+ LSE*log2e and -D by bulk copy) into one of two slots, one barrier each.
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
// Shared memory: K, V (one item), Q and dO (two slots each, 128-byte swizzle), LSE*log2e and -D
// (per slot), barriers, and two item buffers (bitmap row of the backward bitmap, item description;
// the non-empty query tiles are found by scanning the row), and a staging tile through which the
// item's dV and then dK leave: once every MMA of the item is done the compute warps read them
// from TMEM, write them there in the layout of a TMA load, and one thread stores the tile with
// TMA.  The next item's first MMA waits only for the compute warps to have read the
// accumulators.
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
  // an item's dV, then its dK, on their way out (bf16, laid out for the TMA store)
  static constexpr uint32_t kStage = 6 * kTileBytes;
  static constexpr uint32_t kLse2 = 7 * kTileBytes;    // [2 slots][128 floats]: -LSE * log2(e)
  static constexpr uint32_t kDelta = kLse2 + 1024u;    // [2 slots][128 floats]: -D
  static constexpr uint32_t kBar = kDelta + 1024u;
  // per item (two buffers): the bitmap row (at most 64 words, NT <= 1024) and the item's
  // description {b << 16 | k_tile (or -1 for an invalid schedule entry), head, tile count}
  static constexpr uint32_t kRow = kBar + 256u;
  static constexpr uint32_t kInfo = kRow + 2u * 256u;
  static constexpr uint32_t kTotal = kInfo + 32u;
  // no alignment slack: dynamic shared memory starts on a 1024-byte boundary here (no static
  // shared memory); the kernel checks it and reports a device check failure otherwise
  static constexpr uint32_t kAlloc = kTotal;
};
static_assert(Smem<128>::kAlloc <= 232448, "backward shared memory exceeds 227 KB");

enum {
  B_KV = 0,        // K and V of the item loaded
  B_QFULL = 1,     // +slot: Q, dO, LSE*log2e and D of a query tile loaded (one barrier: each
                   // wait of the MMA thread leaves a gap in the tensor pipe)
  B_QEMPTY = 3,    // +slot: the dK MMA (last reader of the slot, after dV) is done
  B_SFULL = 5,     // S^T of the current tile computed
  B_DPFULL = 6,    // dP^T of the current tile computed
  B_PDS = 7,       // compute warps wrote dS^T (TMEM) and read dP^T (8 arrivals)
  B_DONE = 8,      // every MMA of the item completed (dK, dV final)
  B_PREADY = 9,    // compute warps wrote P^T (TMEM) (8 arrivals)
  B_DRAIN = 10,    // abort path only: every MMA issued so far has completed
  B_KVEMPTY = 11,  // the item's last S^T and dP^T MMAs (the last readers of K and V) are done
  B_ACCFREE = 12,  // the compute warps have read the item's dV and dK (8 arrivals)
  B_ROWFULL = 13,  // +buffer: the producer staged an item's bitmap row and description
  B_ROWEMPTY = 15, // +buffer: its readers are done with it (8 compute warps + the MMA thread)
  B_SDV = 17,      // the compute warps wrote the item's dV into the staging tile (8 arrivals)
  B_SDK = 18,      // ... and then its dK (8 arrivals)
  B_SFREE = 19,    // the TMA store of the staging tile has read it (twice per item: dV, dK)
  B_COUNT = 20
};
static_assert(8 * B_COUNT + 8 <= 256, "backward barrier area");


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
                const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                const __grid_constant__ BwdParams p) {
  using L = Smem<D>;
  constexpr int kHalf = D / 2;           // head-dim columns per compute warp
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  int* const queue = p.status + 2 + 2 * (p.NT + 1) + 2;  // work queue (mask.cuh)
  if ((sbase & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment (see Smem)
    if (threadIdx.x == 0) set_status(p.status, kDevBadMeta, 0x2ff);
    if (threadIdx.x == 0) queue_finish(queue);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * B_COUNT + 4);
  int4* info = reinterpret_cast<int4*>(smem + L::kInfo);  // [2]
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const WaitCtl wait{abort_flag, p.status, p.wait_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = p.B * p.NT * p.H;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_KV), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(B_QFULL + x), 1);
      mbar_init(bar(B_QEMPTY + x), 1);
      mbar_init(bar(B_ROWFULL + x), 1);
      mbar_init(bar(B_ROWEMPTY + x), kComputeWarps + 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_DPFULL), 1);
    mbar_init(bar(B_PDS), kComputeWarps);
    mbar_init(bar(B_DONE), 1);
    mbar_init(bar(B_PREADY), kComputeWarps);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_KVEMPTY), 1);
    mbar_init(bar(B_ACCFREE), kComputeWarps);
    mbar_init(bar(B_SDV), kComputeWarps);
    mbar_init(bar(B_SDK), kComputeWarps);
    mbar_init(bar(B_SFREE), 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // asynchronous work issued so far, for the abort path: K/V loads and query-tile slots armed
  // (producer), any MMA issued (MMA thread)
  int kv_armed = 0, g_armed = 0;
  bool mma_issued = false;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
    }
    bool ok = true;
    int gbase = 0;
    for (int k = 0; ok; ++k) {
      const int rb = k & 1;
      // the row buffer is free once its readers are done with item k - 2
      if (k >= 2) {
        const bool free_ = wait(bar(B_ROWEMPTY + rb), ((k >> 1) - 1) & 1, 0x200);
        __syncwarp();
        if (!free_) { ok = false; break; }
      }
      // the next work item from the queue (schedule order: longest rows first); the end
      // marker stops every role
      int jj = 0;
      if (lane == 0) jj = atomicAdd(queue, 1);
      jj = __shfl_sync(0xFFFFFFFFu, jj, 0);
      if (jj >= n_items) {
        if (lane == 0) {
          info[rb] = make_int4(-1, 0, 0, 1);
          mbar_arrive(bar(B_ROWFULL + rb));
        }
        break;
      }
      int item_idx, h;  // head-grouped chunks of the schedule (L2 locality, longest rows first)
      cta_work(jj, n_items / p.H, p.H, item_idx, h);
      const int item = p.sched[item_idx];
      const int b = item >> 16, kt = item & 0xFFFF;
      const bool valid = b >= 0 && b < p.B && kt < p.NT;
      uint32_t* row = reinterpret_cast<uint32_t*>(smem + L::kRow + rb * 256u);
      int cnt = 0;
      if (valid) {
        const uint32_t* src = p.bm + (static_cast<size_t>(b) * p.NT + kt) * p.W;
        for (int w = lane; w < p.W; w += 32) {
          const uint32_t x = src[w];
          row[w] = x;
          cnt += __popc((x | (x >> 1)) & 0x55555555u);
        }
      }
      cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
      if (lane == 0) {
        if (!valid) set_status(p.status, kDevBadSchedule, item_idx);  // nothing is computed
        info[rb] = make_int4(valid ? item : -1, h, cnt, 0);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ROWFULL + rb));
      if (lane == 0 && cnt > 0) {
        const int row0 = (b * p.H + h) * p.S;
        // K and V of this item once the previous item's last S^T and dP^T are done
        if (kv_armed > 0 && !wait(bar(B_KVEMPTY), (kv_armed - 1) & 1, 0x201)) ok = false;
        if (ok) {
          ++kv_armed;
          mbar_arrive_expect_tx(bar(B_KV), 2 * L::kTileBytes);
          for (int x = 0; x < D / 64; ++x) {
            tma_load_2d(sbase + L::kK + x * 16384u, &tmK, x * 64, row0 + kt * 128, bar(B_KV));
            tma_load_2d(sbase + L::kV + x * 16384u, &tmV, x * 64, row0 + kt * 128, bar(B_KV));
          }
        }
        int qt = next_tile(row, p.NT, 0);
        for (int m = 0; ok && m < cnt; ++m, qt = next_tile(row, p.NT, qt + 1)) {
          const int g = gbase + m, slot = g & 1;
          const size_t r = static_cast<size_t>(row0) + qt * 128;
          // a slot is free once the dK MMA of the tile two back (its last reader) is done
          if (g >= 2 && !wait(bar(B_QEMPTY + slot), ((g - 2) >> 1) & 1, 0x202)) {
            ok = false;
            break;
          }
          const uint32_t full = bar(B_QFULL + slot);
          g_armed = g + 1;
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
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      gbase += cnt;
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = make_idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
      constexpr uint32_t idKM = make_idesc_bf16(128, D, 0, 1);    // dK, dV
      const uint32_t sK = sbase + L::kK, sV = sbase + L::kV;
      // low words of the shared-memory descriptors (the split form keeps the issue loop short:
      // the issuing thread shares its SM sub-partition with two compute warps, and every
      // instruction it needs between MMAs leaves the tensor pipe waiting longer)
      const uint32_t dK0 = sdesc_lo(sK, 16u), dV0 = sdesc_lo(sV, 16u);
      // S^T(g) = K Q(g)^T -> region X(g) (g even: RA, odd: RB); dP^T(g) = V dO(g)^T -> X(g + 1)
      // first: the first tile of an item.  For the others the compute warps saw Q and dO of the
      // tile land before their PDS arrival, which this thread has waited for: one wait less in
      // the issue loop (each costs the tensor pipe a gap)
      auto issue_st = [&](int g, bool first) -> bool {
        const int slot = g & 1;
        if (first && !wait(bar(B_QFULL + slot), (g >> 1) & 1, 0x203)) return false;
        tc_fence_after();
        mma_issued = true;
        const uint32_t X = slot ? kColRB : kColRA;
        const uint32_t dQn = sdesc_lo(sbase + L::kQ + slot * L::kTileBytes, 16u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_lo(tmem + X, dK0 + kstep_kmajor(kk), dQn + kstep_kmajor(kk), idSS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL));
        return true;
      };
      auto issue_dpt = [&](int g) {  // its dO landed with its Q (waited for before S^T(g))
        const int slot = g & 1;
        const uint32_t Y = slot ? kColRA : kColRB;
        const uint32_t ddOn = sdesc_lo(sbase + L::kdO + slot * L::kTileBytes, 16u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_lo(tmem + Y, dV0 + kstep_kmajor(kk), ddOn + kstep_kmajor(kk), idSS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_DPFULL));
      };
      bool ok = true;
      int gbase = 0, kq = 0;  // query tiles and computed items before the current one
      for (int k = 0; ok; ++k) {
        const int rb = k & 1;
        if (!wait(bar(B_ROWFULL + rb), (k >> 1) & 1, 0x204)) break;
        if (info[rb].w) break;  // no more work items
        const int nt = info[rb].z;
        mbar_arrive(bar(B_ROWEMPTY + rb));
        if (nt == 0) continue;
        // the first tile: S^T and dP^T as soon as this item's K and V landed
        ok = wait(bar(B_KV), kq & 1, 0x205) && issue_st(gbase, true);
        if (!ok) break;
        issue_dpt(gbase);
        if (nt == 1) umma_commit(bar(B_KVEMPTY));  // no further reader of K and V
        for (int m = 0; ok && m < nt; ++m) {
          const int g = gbase + m, slot = g & 1;
          const uint32_t X = slot ? kColRB : kColRA;
          const uint32_t sQ = sbase + L::kQ + slot * L::kTileBytes;
          const uint32_t sdO = sbase + L::kdO + slot * L::kTileBytes;
          // dV += P^T dO as soon as P^T is in X, while the compute warps work on dS^T.
          // P^T pairs: queries [0,64) at X columns [0,32), [64,128) at [64,96).  The first dV of
          // an item overwrites the accumulator once the compute warps have read the previous one.
          if (!wait(bar(B_PREADY), g & 1, 0x206) ||
              (m == 0 && kq >= 1 && !wait(bar(B_ACCFREE), (kq - 1) & 1, 0x207))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts_lo(tmem + kColDV, tmem + X + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                       sdesc_lo(sdO, 16384u) + kstep_mnmajor(kk), idKM, (m > 0 || kk > 0) ? 1u : 0u);
          if (!wait(bar(B_PDS), g & 1, 0x208)) { ok = false; break; }
          tc_fence_after();
          // the next tile's S^T into Y (its dP^T was consumed), so that its P can start while
          // the tensor pipe runs dK
          if (m + 1 < nt && !issue_st(g + 1, false)) { ok = false; break; }
          // dK += dS^T Q with dS^T read from X: queries [64h + 32c, +32) at columns 64h + 32 + 16c
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts_lo(tmem + kColDK, tmem + X + 64 * (kk >> 2) + 32 + 8 * (kk & 3),
                       sdesc_lo(sQ, 16384u) + kstep_mnmajor(kk), idKM, (m > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(B_QEMPTY + slot));
          if (m + 1 < nt) {
            // dP^T of the next tile into X, after dV and dK above have read P^T and dS^T from it
            issue_dpt(g + 1);
            if (m + 2 == nt) umma_commit(bar(B_KVEMPTY));  // the item's last S^T and dP^T
          }
        }
        if (ok) umma_commit(bar(B_DONE));
        gbase += nt;
        ++kq;
      }
    }
  } else {
    // ---------------------------------------------------------------- compute warps 0-7
    const int quarter = warp & 3;
    const int hf = warp >> 2;
    const int r = quarter * 32 + lane;  // key row (S^T, dP^T, dV, dK)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int gbase = 0, kq = 0;
    int ne = 0;  // items whose dV and dK went out through the staging tile
    // An item's description and this key column's intervals are fetched one item ahead, so that
    // the global loads overlap the previous item's epilogue.
    struct Item {
      int4 it;
      RowIntervals<MAXNI> ri;
    };
    auto fetch = [&](int kf, Item& x) -> bool {
      const bool ready = wait(bar(B_ROWFULL + (kf & 1)), (kf >> 1) & 1, 0x210);
      __syncwarp();
      if (!ready) return false;
      x.it = info[kf & 1];
      if (x.it.x >= 0)
        load_row_intervals(p.itab, x.it.x >> 16, p.NI, p.S, (x.it.x & 0xFFFF) * 128 + r, x.ri);
      return true;
    };
    Item cur;
    cur.it = make_int4(-1, 0, 0, 0);
    ok = fetch(0, cur);
    for (int k = 0; ok && cur.it.w == 0; ++k) {
      const int rb = k & 1;
      const uint32_t* bmrow = reinterpret_cast<const uint32_t*>(smem + L::kRow + rb * 256u);
      const int nt = cur.it.z;
      const int b = cur.it.x >> 16, kt = cur.it.x & 0xFFFF, h = cur.it.y;
      const int row0 = (b * p.H + h) * p.S;
      const int j = kt * 128 + r;  // key column owned for S^T / dP^T
      if (warp == 0 && h == 0 && cur.it.x >= 0) {
        // The backward descriptor must describe the transposed mask of the forward one: tile
        // (kt, q) of this bitmap row has the state of tile (q, kt) of the forward bitmap.
        // Checked once per key tile (head 0); a mismatch (two MaskSpecs that do not describe the
        // same mask) is recorded in the status word, the computation goes on.
        bool bad = false;
        for (int q = lane; q < p.NT; q += 32) {
          const uint32_t cb = (bmrow[q >> 4] >> (2 * (q & 15))) & 3u;
          const uint32_t cf =
              (p.bm_f[(static_cast<size_t>(b) * p.NT + q) * p.W + (kt >> 4)] >> (2 * (kt & 15))) & 3u;
          bad |= cb != cf;
        }
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_status(p.status, kDevDescMismatch, kt);
      }
      int qt = next_tile(bmrow, p.NT, 0);
      for (int m = 0; m < nt; ++m, qt = next_tile(bmrow, p.NT, qt + 1)) {
        const int g = gbase + m, slot = g & 1;
        const bool full = tile_is_full(bmrow, qt);
        const uint32_t X = slot ? kColRB : kColRA;
        const uint32_t Y = slot ? kColRA : kColRB;

        // ---- P^T: S^T from X, written back in place as bf16 pairs; fp32 P kept for dS ----
        bool ready = wait(bar(B_SFULL), g & 1, 0x211) &&
                     wait(bar(B_QFULL + slot), (g >> 1) & 1, 0x212);
        __syncwarp();
        if (!ready) { ok = false; break; }
        tc_fence_after();
        float pf[2][32];
        const uint32_t lse2_base = sbase + L::kLse2 + slot * 512u;
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
            const uint32_t vis = visible_bits_any(i0, cur.ri, p.NI, p.check, p.masked != 0);
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
        ready = wait(bar(B_DPFULL), g & 1, 0x213);
        __syncwarp();
        if (!ready) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int q0 = 64 * hf + 32 * ch;
          uint32_t dpr[32], dd[16];
          tmem_ld32(tmem + lane_off + Y + q0, dpr);
          tmem_wait_ld();
          ds_chunk(pf[ch], dpr, sbase + L::kDelta + slot * 512u + q0 * 4u, dd);
          // dS^T pairs into X columns this warp has read and P^T does not use: 64 hf + 32 + 16 ch
          tmem_st16(tmem + lane_off + X + hf * 64 + 32 + ch * 16, dd);
        }
        tmem_wait_st();
        tc_fence_before();
        // the next tile's Q and dO have landed (the MMA thread relies on it for S^T(g+1))
        if (m + 1 < nt) {
          ready = wait(bar(B_QFULL + (slot ^ 1)), ((g + 1) >> 1) & 1, 0x218);
          __syncwarp();
          if (!ready) { ok = false; break; }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PDS));
      }
      // the bitmap row and the item description are no longer needed
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ROWEMPTY + rb));
      if (!ok) break;
      const Item done_item = cur;
      if (!fetch(k + 1, cur)) { ok = false; break; }  // (the producer stages an end marker last)
      if (done_item.it.x < 0) continue;  // an invalid schedule entry: nothing to write
      __nv_bfloat16* dvrow = p.dv + (static_cast<size_t>(row0) + j) * D + hf * kHalf;
      __nv_bfloat16* dkrow = p.dk + (static_cast<size_t>(row0) + j) * D + hf * kHalf;
      if (nt == 0) {  // a key tile that no query sees
        uint4* dva = reinterpret_cast<uint4*>(dvrow);
        uint4* dka = reinterpret_cast<uint4*>(dkrow);
        for (int q = 0; q < kHalf / 8; ++q) {
          dva[q] = make_uint4(0, 0, 0, 0);
          dka[q] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      // ---- epilogue: dV, dK (scaled) -> bf16, this warp's half of the head dim ----
      const bool fin = wait(bar(B_DONE), kq & 1, 0x214);
      __syncwarp();
      if (!fin) { ok = false; break; }
      tc_fence_after();
      const float sc = p.scale;
      uint32_t ob[2][kHalf / 2];  // dV, then dK (scaled), as bf16 pairs of this row's columns
#pragma unroll
      for (int x = 0; x < 2; ++x) {
#pragma unroll
        for (int c = 0; c < kHalf; c += 32) {
          uint32_t a[32];
          tmem_ld32(tmem + lane_off + (x == 0 ? kColDV : kColDK) + hf * kHalf + c, a);
          tmem_wait_ld();
          const float f = x == 0 ? 1.f : sc;
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            ob[x][(c + e) / 2] = pack_bf16x2(__uint_as_float(a[e]) * f, __uint_as_float(a[e + 1]) * f);
        }
      }
      // the accumulators are free for the next item
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ACCFREE));
      // dV, then dK, leave through the staging tile: each warp writes its rows and columns there,
      // one thread stores the tile with TMA.  The stores run on while the next item starts; the
      // tile is rewritten once the previous store has read it.
      const bool storer = warp == 0 && lane == 0;
      const uint32_t stg = sbase + L::kStage;
      for (int x = 0; x < 2 && ok; ++x) {
        const int step = 2 * ne + x;  // stores through the staging tile so far
        if (step > 0) {
          if (storer) {
            bulk_wait_read_all();
            mbar_arrive(bar(B_SFREE));
          }
          const bool free_ = wait(bar(B_SFREE), (step - 1) & 1, 0x215);
          __syncwarp();
          if (!free_) { ok = false; break; }
        }
        const uint32_t box = stg + (D == 128 ? hf * 16384u : 0u);
        const int c0 = D == 128 ? 0 : hf * (kHalf / 8);
#pragma unroll
        for (int c = 0; c < kHalf / 8; ++c)
          st_shared_v4(swz128_chunk(box, r, c0 + c), ob[x][4 * c], ob[x][4 * c + 1], ob[x][4 * c + 2],
                       ob[x][4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(x == 0 ? B_SDV : B_SDK));
        if (storer) {
          if (!wait(bar(x == 0 ? B_SDV : B_SDK), ne & 1, 0x216)) { ok = false; break; }
          for (int bx = 0; bx < D / 64; ++bx)
            tma_store_2d(x == 0 ? &tmdV : &tmdK, bx * 64, row0 + kt * 128, stg + bx * 16384u);
          bulk_commit_group();
        }
      }
      ++ne;
      gbase += nt;
      ++kq;
    }
    // the last TMA stores complete before the CTA exits (and its shared memory goes)
    if (warp == 0 && lane == 0) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up.  Copies and MMAs already issued still land in shared memory and TMEM:
    // wait for them before TMEM is freed and the CTA exits.
    if (warp == kProducerWarp && lane == 0) {
      if (kv_armed > 0) mbar_wait_drain(bar(B_KV), (kv_armed - 1) & 1, p.status, 0x2f0);
      for (int g = g_armed - 2; g < g_armed; ++g)
        if (g >= 0) mbar_wait_drain(bar(B_QFULL + (g & 1)), (g >> 1) & 1, p.status, 0x2f1);
    }
    if (warp == kMmaWarp && lane == 0 && mma_issued) {
      umma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0, p.status, 0x2f2);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (threadIdx.x == 0) queue_finish(queue);
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
int bwd_launch(dim3 grid, cudaStream_t stream, const CUtensorMap& mq, const CUtensorMap& mk,
               const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mdk,
               const CUtensorMap& mdv, const BwdParams& p) {
  const uint32_t smem = bwd::Smem<D>::kAlloc;
  if (cudaFuncSetAttribute(bwd::attn_bwd_kernel<D, MAXNI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -1;
  bwd::attn_bwd_kernel<D, MAXNI><<<grid, bwd::kThreads, smem, stream>>>(mq, mk, mv, mdo, mdk, mdv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_attn_dkdv(const BwdParams& p, int d, const void* q, const void* k, const void* v,
                     const void* d_o, cudaStream_t stream) {
  const size_t rows = static_cast<size_t>(p.B) * p.H * p.S;
  CUtensorMap mq, mk, mv, mdo, mdk, mdv;
  if (!make_bf16_tile_map(&mq, q, rows, d) || !make_bf16_tile_map(&mk, k, rows, d) ||
      !make_bf16_tile_map(&mv, v, rows, d) || !make_bf16_tile_map(&mdo, d_o, rows, d) ||
      !make_bf16_tile_map(&mdk, p.dk, rows, d) || !make_bf16_tile_map(&mdv, p.dv, rows, d))
    return -1;
  // persistent: one CTA per SM (one fits: 227 KB of shared memory, all 512 TMEM columns)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return -1;
  const int items = p.B * p.NT * p.H;
  const dim3 grid(items < sms ? items : sms);
  // interval registers: 4 cover every visible-form workload here; 9 the largest tables
  if (d == 128) {
    if (p.NI <= 4) return bwd_launch<128, 4>(grid, stream, mq, mk, mv, mdo, mdk, mdv, p);
    return bwd_launch<128, 9>(grid, stream, mq, mk, mv, mdo, mdk, mdv, p);
  }
  if (p.NI <= 4) return bwd_launch<64, 4>(grid, stream, mq, mk, mv, mdo, mdk, mdv, p);
  return bwd_launch<64, 9>(grid, stream, mq, mk, mv, mdo, mdk, mdv, p);
}

}  // namespace cm

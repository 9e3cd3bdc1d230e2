// Descriptor-guided attention, backward (CompileMask sections 3.2.2 / 3.3 / 3.3.2), for sm_103a.
//
// The backward pass traverses key tiles, so it uses the backward descriptor: per key column j,
// the visible query intervals, and per (key tile, query tile) the 2-bit state.  One CTA owns one
// 128-key tile of one (sample, head) and walks the non-empty query tiles of its bitmap row:
//
//   S^T  = K Q^T            (tcgen05, TMEM)        P^T  = exp2(S^T * scale*log2e - LSE*log2e)
//   dP^T = V dO^T           (tcgen05, TMEM)        dS^T = P^T * (dP^T - D),  D = rowsum(dO * O)
//   dK  += dS^T Q           (TMEM accumulator)
//   dV  += P^T dO           (TMEM accumulator; P^T is the A operand, read from TMEM)
//   dQ_part = dS K          (TMEM) -> shared memory -> TMA bulk add into the fp32 dQ accumulator
//
// Partial tiles check each query index against the key column's intervals with the unsigned
// test of section 4.4 and zero P there (the -inf of the forward); full tiles skip the check.
// Empty tiles are never visited.
//
// Warp roles (320 threads):
//   warps 0-7  compute.  Warp w serves TMEM lane quarter w % 4 (key rows 32*(w%4) ..) and column
//              half w / 4: queries [64*half, +64) of S^T / dP^T, and head-dim columns
//              [half*d/2, +d/2) of dQ_part, dV and dK.
//   warp 8     TMA producer: K, V once; per query tile Q (+ LSE*log2e by bulk copy) and dO (+ D).
//   warp 9     MMA issuer (one thread).  Per query tile: S^T, dP^T; then dK (its completion
//              frees Q for the next tile), dV (frees dO), and dQ_part.
// TMEM (512 columns): dV [0, d), dK [128, 128+d), R1 [256, 384) = S^T, overwritten in place by
// the bf16 P^T pairs (each warp writes only columns it has already read), R2 [384, 512) = dP^T,
// then dQ_part.
// Shared memory: K, V, Q, dO, dS^T (bf16, 128-byte swizzle), one 16 KB fp32 staging tile per
// column half for the dQ bulk add, LSE*log2e and D of the current query tile.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace cm {

namespace bwd {

constexpr int kComputeWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kMaxTiles = 1024;

constexpr uint32_t kColDV = 0;
constexpr uint32_t kColDK = 128;
constexpr uint32_t kColR1 = 256;
constexpr uint32_t kColR2 = 384;

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Smem {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kTileBytes;
  static constexpr uint32_t kQ = 2 * kTileBytes;
  static constexpr uint32_t kdO = 3 * kTileBytes;
  static constexpr uint32_t kdSt = 4 * kTileBytes;   // [2 boxes][128 keys][64 queries] bf16
  static constexpr uint32_t kStage = kdSt + 32768u;  // fp32 [2 halves][128 rows][32 cols]
  static constexpr uint32_t kLse2 = kStage + 32768u; // 128 floats: -LSE * log2(e)
  static constexpr uint32_t kDelta = kLse2 + 512u;   // 128 floats: -D
  static constexpr uint32_t kBar = kDelta + 512u;
  static constexpr uint32_t kList = kBar + 256u;
  static constexpr uint32_t kTotal = kList + 2u * kMaxTiles;
  static constexpr uint32_t kAlloc = kTotal + 1024u;
};

enum {
  B_KV = 0,       // K and V loaded
  B_QFULL = 1,    // Q and LSE*log2e of the current query tile loaded
  B_QEMPTY = 2,   // the dK MMA (last reader of Q) of the current tile is done
  B_DOFULL = 3,   // dO and D of the current query tile loaded
  B_DOEMPTY = 4,  // the dV MMA (last reader of dO) of the current tile is done
  B_SFULL = 5,    // S^T and dP^T computed
  B_PDS = 6,      // compute warps wrote P^T (TMEM) and dS^T (smem) (8 arrivals)
  B_DQFULL = 7,   // dQ_part computed (and every MMA of the tile done)
  B_DQREAD = 8,   // compute warps read dQ_part from TMEM (8 arrivals)
  B_STGFREE = 9,  // +half: the half's staging tile may be written (its leader, 1 arrival)
  B_STGFULL = 11, // +half: the half's 4 warps wrote their staging rows (4 arrivals)
  B_COUNT = 13
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

template <int NI>
__device__ __forceinline__ uint32_t visible_bits(int i0, const int (&st)[4], const uint32_t (&len)[4]) {
  // bit c set iff query i0 + c (c < 32) lies in one of the column's intervals
  uint32_t bits = 0;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    bool vis = false;
#pragma unroll
    for (int n = 0; n < NI; ++n)
      vis |= (static_cast<uint32_t>(i0 - st[n]) + static_cast<uint32_t>(c)) < len[n];
    bits |= vis ? (1u << c) : 0u;
  }
  return bits;
}

// P^T and dS^T of 32 queries of this key row.  For a full tile every query is visible; for a
// partial tile `vis` holds the visibility bits.
template <bool FULL>
__device__ __forceinline__ void chunk_p_ds(const uint32_t (&sr)[32], const uint32_t (&dpr)[32],
                                           uint32_t lse2_addr, uint32_t delta_addr, float sl2,
                                           uint32_t vis, uint32_t (&pp)[16], uint32_t (&dd)[16]) {
  // shared memory holds -LSE*log2e and -D per query, so both steps are paired FMAs / adds:
  // x = s * scale*log2e + (-lse2),  p = exp2(x),  g = dp + (-D),  ds = p * g
  const float2 scale2 = make_float2(sl2, sl2);
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const float4 l4 = ld_shared_f4(lse2_addr + c * 4u);
    const float4 d4 = ld_shared_f4(delta_addr + c * 4u);
    const float2 xa = fma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), scale2,
                           make_float2(l4.x, l4.y));
    const float2 xb = fma2(make_float2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])),
                           scale2, make_float2(l4.z, l4.w));
    float2 pa = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
    float2 pb = make_float2(ex2_approx(xb.x), ex2_approx(xb.y));
    if (!FULL) {
      pa.x = ((vis >> c) & 1u) ? pa.x : 0.f;
      pa.y = ((vis >> (c + 1)) & 1u) ? pa.y : 0.f;
      pb.x = ((vis >> (c + 2)) & 1u) ? pb.x : 0.f;
      pb.y = ((vis >> (c + 3)) & 1u) ? pb.y : 0.f;
    }
    const float2 ga = add2(make_float2(__uint_as_float(dpr[c]), __uint_as_float(dpr[c + 1])),
                           make_float2(d4.x, d4.y));
    const float2 gb = add2(make_float2(__uint_as_float(dpr[c + 2]), __uint_as_float(dpr[c + 3])),
                           make_float2(d4.z, d4.w));
    const float2 dsa = mul2(pa, ga);
    const float2 dsb = mul2(pb, gb);
    pp[c / 2] = pack_bf16x2(pa.x, pa.y);
    pp[c / 2 + 1] = pack_bf16x2(pb.x, pb.y);
    dd[c / 2] = pack_bf16x2(dsa.x, dsa.y);
    dd[c / 2 + 1] = pack_bf16x2(dsb.x, dsb.y);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ BwdParams p) {
  using L = Smem<D>;
  constexpr int kHalf = D / 2;           // head-dim columns per compute warp
  constexpr int kChunks = kHalf / 32;    // 32-column dQ chunks per warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * B_COUNT + 4);
  int* s_ntiles = reinterpret_cast<int*>(smem + L::kBar + 8 * B_COUNT + 8);
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int item = p.sched[blockIdx.x / p.H];
  const int h = blockIdx.x % p.H;
  const int b = item >> 16;
  const int kt = item & 0xFFFF;
  const int bh = b * p.H + h;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_KV), 1);
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_DOFULL), 1);
    mbar_init(bar(B_DOEMPTY), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_PDS), kComputeWarps);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQREAD), kComputeWarps);
    for (int hh = 0; hh < 2; ++hh) {
      mbar_init(bar(B_STGFREE + hh), 1);
      mbar_init(bar(B_STGFULL + hh), 4);
    }
    fence_barrier_init();
  }
  if (warp == 0) {
    const uint32_t* row = p.bm + (static_cast<size_t>(b) * p.NT + kt) * p.W;
    int base = 0;
    for (int c0 = 0; c0 < p.NT; c0 += 32) {
      const int c = c0 + lane;
      uint32_t code = 0;
      if (c < p.NT) code = (row[c >> 4] >> (2 * (c & 15))) & 3u;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, code != 0);
      if (code != 0)
        list[base + __popc(m & ((1u << lane) - 1u))] =
            static_cast<uint16_t>(c | (code == 2u ? 0x8000 : 0));
      base += __popc(m);
    }
    if (lane == 0) *s_ntiles = base;
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

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      tma_prefetch_desc(&tmdQ);
      mbar_arrive_expect_tx(bar(B_KV), 2 * L::kTileBytes);
      for (int x = 0; x < D / 64; ++x) {
        tma_load_2d(sbase + L::kK + x * 16384u, &tmK, x * 64, row0 + kt * 128, bar(B_KV));
        tma_load_2d(sbase + L::kV + x * 16384u, &tmV, x * 64, row0 + kt * 128, bar(B_KV));
      }
      for (int m = 0; m < nt; ++m) {
        const int qt = list[m] & 0x3FFF;
        const size_t r = static_cast<size_t>(row0) + qt * 128;
        // Q is free once the previous tile's dK MMA is done, dO once its dV MMA is done
        if (m >= 1 && !mbar_wait(bar(B_QEMPTY), (m - 1) & 1, abort_flag, p.status, 0x201)) break;
        mbar_arrive_expect_tx(bar(B_QFULL), L::kTileBytes + 512u);
        for (int x = 0; x < D / 64; ++x)
          tma_load_2d(sbase + L::kQ + x * 16384u, &tmQ, x * 64, row0 + qt * 128, bar(B_QFULL));
        bulk_load(sbase + L::kLse2, p.lse2 + r, 512u, bar(B_QFULL));
        if (m >= 1 && !mbar_wait(bar(B_DOEMPTY), (m - 1) & 1, abort_flag, p.status, 0x20b)) break;
        mbar_arrive_expect_tx(bar(B_DOFULL), L::kTileBytes + 512u);
        for (int x = 0; x < D / 64; ++x)
          tma_load_2d(sbase + L::kdO + x * 16384u, &tmdO, x * 64, row0 + qt * 128, bar(B_DOFULL));
        bulk_load(sbase + L::kDelta, p.delta + r, 512u, bar(B_DOFULL));
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idSS = make_idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
      constexpr uint32_t idKM = make_idesc_bf16(128, D, 0, 1);    // dK, dV (TS)
      constexpr uint32_t idMM = make_idesc_bf16(128, D, 1, 1);    // dQ_part
      const uint32_t sK = sbase + L::kK, sV = sbase + L::kV, sQ = sbase + L::kQ,
                     sdO = sbase + L::kdO, sdSt = sbase + L::kdSt;
      bool ok = mbar_wait(bar(B_KV), 0, abort_flag, p.status, 0x202);
      for (int m = 0; ok && m < nt; ++m) {
        if (!mbar_wait(bar(B_QFULL), m & 1, abort_flag, p.status, 0x203)) break;
        if (!mbar_wait(bar(B_DOFULL), m & 1, abort_flag, p.status, 0x20c)) break;
        // dQ_part of the previous tile has been read out of R2, which also means every MMA of the
        // previous tile (including the dV that read P^T from R1) has completed
        if (m >= 1 && !mbar_wait(bar(B_DQREAD), (m - 1) & 1, abort_flag, p.status, 0x204)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColR1, sdesc_kmajor(sK, kk, 16384u), sdesc_kmajor(sQ, kk, 16384u), idSS,
                  kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColR2, sdesc_kmajor(sV, kk, 16384u), sdesc_kmajor(sdO, kk, 16384u), idSS,
                  kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL));
        if (!mbar_wait(bar(B_PDS), m & 1, abort_flag, p.status, 0x205)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + kColDK, sdesc_kmajor(sdSt, kk, 16384u), sdesc_mnmajor(sQ, kk, 16384u), idKM,
                  (m > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(B_QEMPTY));
        // P^T pairs: queries [0,64) at R1 columns [0,32), queries [64,128) at [64,96)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + kColDV, tmem + kColR1 + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                  sdesc_mnmajor(sdO, kk, 16384u), idKM, (m > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(B_DOEMPTY));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + kColR2, sdesc_mnmajor(sdSt, kk, 16384u), sdesc_mnmajor(sK, kk, 16384u), idMM,
                  kk > 0 ? 1u : 0u);
        umma_commit(bar(B_DQFULL));
      }
    }
  } else {
    // ---------------------------------------------------------------- compute warps 0-7
    const int quarter = warp & 3;
    const int hf = warp >> 2;
    const int r = quarter * 32 + lane;  // key row (S^T, dP^T, dV, dK) / query row (dQ_part)
    const int j = kt * 128 + r;         // key column owned for S^T / dP^T
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const bool leader = (quarter == 0 && lane == 0);  // issues this half's bulk adds
    const uint32_t stage = sbase + L::kStage + hf * 16384u;
    int st[4];
    uint32_t len[4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      st[n] = 0;
      len[n] = 0;
      if (n < p.NI) {
        const int2 iv = reinterpret_cast<const int2*>(p.itab)[(static_cast<size_t>(b) * p.NI + n) * p.S + j];
        st[n] = iv.x;
        len[n] = static_cast<uint32_t>(iv.y - iv.x);
      }
    }
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int m = 0; ok && m < nt; ++m) {
      const int entry = list[m];
      const int qt = entry & 0x3FFF;
      const bool full = (entry & 0x8000) != 0;
      bool ready = mbar_wait(bar(B_SFULL), m & 1, abort_flag, p.status, 0x206) &&
                   mbar_wait(bar(B_QFULL), m & 1, abort_flag, p.status, 0x207) &&
                   mbar_wait(bar(B_DOFULL), m & 1, abort_flag, p.status, 0x20d);
      __syncwarp();
      if (!ready) { ok = false; break; }
      tc_fence_after();
      // this warp's 64 queries, in two chunks of 32
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int q0 = 64 * hf + 32 * ch;  // first query of the chunk within the tile
        uint32_t sr[32], dpr[32];
        tmem_ld32(tmem + lane_off + kColR1 + q0, sr);
        tmem_ld32(tmem + lane_off + kColR2 + q0, dpr);
        tmem_wait_ld();
        uint32_t pp[16], dd[16];
        const uint32_t la = sbase + L::kLse2 + q0 * 4u, da = sbase + L::kDelta + q0 * 4u;
        if (full) {
          chunk_p_ds<true>(sr, dpr, la, da, sl2, 0u, pp, dd);
        } else {
          const int i0 = qt * 128 + q0;
          uint32_t vis;
          switch (p.NI) {
            case 1: vis = visible_bits<1>(i0, st, len); break;
            case 2: vis = visible_bits<2>(i0, st, len); break;
            case 3: vis = visible_bits<3>(i0, st, len); break;
            default: vis = visible_bits<4>(i0, st, len); break;
          }
          chunk_p_ds<false>(sr, dpr, la, da, sl2, vis, pp, dd);
        }
        // P^T pairs into R1 columns this warp has already read: hf * 64 + ch * 16
        tmem_st16(tmem + lane_off + kColR1 + hf * 64 + ch * 16, pp);
        // dS^T row r, queries q0..q0+31 = four 16-byte chunks of box hf
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t chunk = ch * 4 + q4;
          const uint32_t off = hf * 16384u + r * 128u + ((chunk ^ (r & 7)) << 4);
          st_shared_v4(sbase + L::kdSt + off, dd[4 * q4], dd[4 * q4 + 1], dd[4 * q4 + 2], dd[4 * q4 + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PDS));

      // dQ_part: query row r of this tile, head-dim columns [hf * kHalf, +kHalf)
      ready = mbar_wait(bar(B_DQFULL), m & 1, abort_flag, p.status, 0x208);
      __syncwarp();
      if (!ready) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < kChunks; ++cc) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + kColR2 + hf * kHalf + cc * 32, v);
        tmem_wait_ld();
        if (cc == kChunks - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_DQREAD));  // R2 may be overwritten now
        }
        // use u of this half's staging tile: wait until the previous bulk add stopped reading it
        const int u = m * kChunks + cc;
        if (leader) {
          bulk_wait_read_all();
          mbar_arrive(bar(B_STGFREE + hf));
        }
        const bool free_ok = mbar_wait(bar(B_STGFREE + hf), u & 1, abort_flag, p.status, 0x209);
        __syncwarp();
        if (!free_ok) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(stage + r * 128u + ((static_cast<uint32_t>(c) ^ (r & 7)) << 4), v[4 * c],
                       v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_STGFULL + hf));
        bool full_ok = true;
        if (leader) {
          full_ok = mbar_wait(bar(B_STGFULL + hf), u & 1, abort_flag, p.status, 0x20a);
          if (full_ok) {
            tma_reduce_add_2d(&tmdQ, hf * kHalf + cc * 32, row0 + qt * 128, stage);
            bulk_commit_group();
          }
        }
        full_ok = __shfl_sync(0xFFFFFFFFu, full_ok, 0);
        if (!full_ok) { ok = false; break; }
      }
    }
    if (leader) bulk_wait_all();
    __syncwarp();

    // ---- epilogue: dV, dK (scaled) -> bf16, this warp's half of the head dim ----
    __nv_bfloat16* dvrow = p.dv + (static_cast<size_t>(row0) + j) * D + hf * kHalf;
    __nv_bfloat16* dkrow = p.dk + (static_cast<size_t>(row0) + j) * D + hf * kHalf;
    if (nt > 0 && ok) {
      // the last DQFULL wait above guarantees every MMA of this CTA has completed
#pragma unroll
      for (int c = 0; c < kHalf; c += 32) {
        uint32_t a[32], k2[32];
        tmem_ld32(tmem + lane_off + kColDV + hf * kHalf + c, a);
        tmem_ld32(tmem + lane_off + kColDK + hf * kHalf + c, k2);
        tmem_wait_ld();
        uint4* dva = reinterpret_cast<uint4*>(dvrow + c);
        uint4* dka = reinterpret_cast<uint4*>(dkrow + c);
        const float sc = p.scale;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 x, y;
          x.x = pack_bf16x2(__uint_as_float(a[8 * q + 0]), __uint_as_float(a[8 * q + 1]));
          x.y = pack_bf16x2(__uint_as_float(a[8 * q + 2]), __uint_as_float(a[8 * q + 3]));
          x.z = pack_bf16x2(__uint_as_float(a[8 * q + 4]), __uint_as_float(a[8 * q + 5]));
          x.w = pack_bf16x2(__uint_as_float(a[8 * q + 6]), __uint_as_float(a[8 * q + 7]));
          y.x = pack_bf16x2(__uint_as_float(k2[8 * q + 0]) * sc, __uint_as_float(k2[8 * q + 1]) * sc);
          y.y = pack_bf16x2(__uint_as_float(k2[8 * q + 2]) * sc, __uint_as_float(k2[8 * q + 3]) * sc);
          y.z = pack_bf16x2(__uint_as_float(k2[8 * q + 4]) * sc, __uint_as_float(k2[8 * q + 5]) * sc);
          y.w = pack_bf16x2(__uint_as_float(k2[8 * q + 6]) * sc, __uint_as_float(k2[8 * q + 7]) * sc);
          dva[q] = x;
          dka[q] = y;
        }
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
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// Per row, negated for the main kernel's paired FMAs: -D = -sum_c dO[c] * O[c] (fp32) and
// -LSE * log2(e) (-inf for a row that sees nothing, so that its P is exp2(-inf) = 0); and a zeroed
// dQ accumulator row.  One warp per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_prologue_kernel(const __nv_bfloat16* o,
                                                           const __nv_bfloat16* d_o,
                                                           const float* lse, float* delta,
                                                           float* lse2, float* dq_acc,
                                                           size_t rows) {
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
  float* z = dq_acc + row * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) z[e] = 0.f;
}

// dQ = bf16(scale * dQ_acc), 8 elements per thread
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* dq_acc, __nv_bfloat16* dq,
                                                         size_t n8, float scale) {
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * t];
  const float4 c = reinterpret_cast<const float4*>(dq_acc)[2 * t + 1];
  uint4 v;
  v.x = pack_bf16x2(a.x * scale, a.y * scale);
  v.y = pack_bf16x2(a.z * scale, a.w * scale);
  v.z = pack_bf16x2(c.x * scale, c.y * scale);
  v.w = pack_bf16x2(c.z * scale, c.w * scale);
  reinterpret_cast<uint4*>(dq)[t] = v;
}

}  // namespace bwd

int launch_attn_bwd(const BwdParams& p, int d, const void* q, const void* k, const void* v,
                    const void* o, const void* d_o, void* dq, cudaStream_t stream) {
  const size_t rows = static_cast<size_t>(p.B) * p.H * p.S;
  // prologue: D, LSE * log2(e) and the zeroed accumulator
  {
    const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
    if (d == 128)
      bwd::bwd_prologue_kernel<128><<<blocks, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), p.lse,
          p.delta, p.lse2, p.dq_acc, rows);
    else
      bwd::bwd_prologue_kernel<64><<<blocks, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), p.lse,
          p.delta, p.lse2, p.dq_acc, rows);
    if (cudaGetLastError() != cudaSuccess) return -1;
  }
  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!make_bf16_tile_map(&mq, q, rows, d) || !make_bf16_tile_map(&mk, k, rows, d) ||
      !make_bf16_tile_map(&mv, v, rows, d) || !make_bf16_tile_map(&mdo, d_o, rows, d) ||
      !make_f32_tile_map(&mdq, p.dq_acc, rows, d))
    return -1;
  const dim3 grid(p.B * p.NT * p.H);
  if (d == 128) {
    const uint32_t smem = bwd::Smem<128>::kAlloc;
    if (cudaFuncSetAttribute(bwd::attn_bwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return -1;
    bwd::attn_bwd_kernel<128><<<grid, bwd::kThreads, smem, stream>>>(mq, mk, mv, mdo, mdq, p);
  } else {
    const uint32_t smem = bwd::Smem<64>::kAlloc;
    if (cudaFuncSetAttribute(bwd::attn_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return -1;
    bwd::attn_bwd_kernel<64><<<grid, bwd::kThreads, smem, stream>>>(mq, mk, mv, mdo, mdq, p);
  }
  if (cudaGetLastError() != cudaSuccess) return -1;
  const size_t n8 = rows * d / 8;
  bwd::dq_convert_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(
      p.dq_acc, static_cast<__nv_bfloat16*>(dq), n8, p.scale);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace cm

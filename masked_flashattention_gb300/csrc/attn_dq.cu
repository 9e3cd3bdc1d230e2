// Descriptor-guided attention, backward, dQ part (CompileMask sections 3.3.2 / 4.4), for sm_103a.
//
// dQ = scale * sum over key tiles of dS K, with dS = P * (dP - D), P = exp(scale * Q K^T - LSE)
// and dP = dO V^T.  The main backward kernel walks key tiles (it owns dK and dV); accumulating dQ
// there would need an fp32 read-modify-write of every (key tile, query tile) partial in L2, and on
// GB300 that traffic limits the whole backward.  This kernel walks query tiles instead, like the
// forward: a work item is one 128-row query tile of one (sample, head); it visits the key tiles of
// the forward bitmap row (empty tiles skipped, full tiles unmasked, partial tiles checked against
// the forward Interval Table), recomputes S and dP, and keeps dQ in TMEM.  It writes dQ once, in
// bf16, with no atomics.
//
// Persistent CTAs: one CTA per SM; its producer warp takes the next work item of the
// longest-first schedule from a work queue (an atomic counter in the descriptor's status
// buffer).  Barrier phases, K/V slots and TMEM buffers run on across items (global tile counter
// g), so the next item's K/V tiles load and its first S MMAs run while the compute warps write
// the previous item's dQ.  The producer also brings the next item's Q and dO tiles into shared
// memory (TMA), from where the compute warps copy them into TMEM at the item boundary.
//
// Q and dO stay in TMEM for a whole item (the compute warps copy their rows there once), so all
// three MMAs of a key tile take their A operand from TMEM and read only K or V from
// shared memory: S = Q K^T, dP = dO V^T, dQ += dS K.
//
// The per-row constants of the backward come from here too: with its rows of dO the compute warps
// load the same rows of O and form D = rowsum(dO * O) (the two warps of a row each sum half the
// columns and exchange the halves), and take -LSE * log2(e) from the forward's LSE.  They use them
// for dS and write them to the workspace, where the dK/dV kernel, queued after this one, reads
// them: no separate pass over O and dO.
//
// Warp roles (352 threads):
//   warps 0-7  compute.  Warp w serves TMEM lane quarter w % 4 (query rows 32*(w%4) ..) and
//              column half w / 4 of each 128-key tile: it reads S, then P = exp2(S *
//              scale*log2e - LSE*log2e) stays in registers while dP is computed into the same
//              TMEM columns, then dS = P * (dP - D) is written back there as bf16 pairs.
//   warp 8     producer: per item, stages the bitmap row in shared memory (the whole warp), then
//              lane 0 loads the item's Q and dO into the staging tiles (one item ahead), and K
//              through a 3-slot ring and V through a 2-slot ring.
//   warps 9-10 MMA issuers, one thread each: the thread of warp 9 + t issues S(g), dP(g) and
//              dQ(g) of the key tiles g with g % 2 == t.  A thread that issues tcgen05 MMAs
//              stalls on every barrier wait, and the tensor pipe holds too few queued 128 x 128
//              MMAs to cover the stall: with two issuers one thread's MMAs run while the other
//              waits.
// TMEM (512 columns): X0 [0,128), X1 [128,256) (key tile g uses X(g % 2) for S(g), then dP(g),
// then dS(g)), dQ [256, 256+d), Q [384, 384+d/2), dO [448, 448+d/2).  Buffer X(t) belongs to the
// tiles of issuer t, which rewrites it only with MMAs issued after the ones that read it
// (tcgen05 MMAs of one thread run in issue order).  The compute warps store the next item's Q and
// dO once they have read the current item's last dP (every S and dP MMA of the item is then
// done), and the first dQ MMA of an item overwrites dQ once they have read the previous one.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "kernels.h"
#include "mask.cuh"
#include "ptx.cuh"
#include "tma_host.h"

namespace cm {
namespace dq {

constexpr int kComputeWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;  // and 10
constexpr int kThreads = 352;
constexpr int kKStages = 3;
constexpr int kVStages = 2;

constexpr uint32_t kColX = 0;  // + 128 * (n % 2)
constexpr uint32_t kColDQ = 256;
constexpr uint32_t kColQ = 384;
constexpr uint32_t kColDO = 448;

// Dynamic shared memory starts on a 1024-byte boundary here (no static shared memory); the kernel
// checks it and reports a device check failure otherwise.
template <int D>
struct Smem {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kK = 0;                                 // kKStages slots
  static constexpr uint32_t kV = kK + kKStages * kTileBytes;        // kVStages slots
  // the next item's Q and dO tiles (TMA, 128-byte swizzle), copied into TMEM by the compute warps
  static constexpr uint32_t kQS = kV + kVStages * kTileBytes;
  static constexpr uint32_t kdOS = kQS + kTileBytes;
  static constexpr uint32_t kBar = kdOS + kTileBytes;
  // per item (two buffers): the bitmap row (at most 64 words, NT <= 1024) and the item's
  // description {b << 16 | q_tile (or -1 for an invalid schedule entry), head, tile count}
  static constexpr uint32_t kRow = kBar + 512u;
  static constexpr uint32_t kInfo = kRow + 2u * 256u;
  // halves of D = rowsum(dO * O), exchanged by the two warps of a row: [2 halves][128 rows]
  static constexpr uint32_t kDPart = kInfo + 32u;
  static constexpr uint32_t kTotal = kDPart + 2u * 128u * 4u;
  static constexpr uint32_t kAlloc = kTotal;
};
static_assert(Smem<128>::kAlloc <= 232448, "dQ kernel shared memory exceeds 227 KB");

enum {
  B_QDO = 0,      // Q and dO of the item stored in TMEM by the compute warps (8 arrivals)
  B_KFULL = 1,    // +slot (3)
  B_KEMPTY = 4,   // +slot (3): the dQ MMA that last read the K slot is done
  B_VFULL = 7,    // +slot (2)
  B_VEMPTY = 9,   // +slot (2): the dP MMA that read the V slot is done
  B_SFULL = 11,   // +buffer (2): S of the buffer's tile computed
  B_SREAD = 13,   // +buffer (2): compute warps hold S in registers (8 arrivals)
  B_DPFULL = 15,  // +buffer (2): dP of the buffer's tile computed
  B_DSFULL = 17,  // +buffer (2): compute warps wrote dS (8 arrivals)
  B_DONE = 19,    // every MMA of the item completed (one commit per issuer per item)
  B_DRAIN = 20,   // +issuer, abort path only: every MMA the issuer issued has completed
  B_DQFREE = 22,  // the compute warps have read the item's dQ (8 arrivals)
  B_ROWFULL = 23, // +buffer: the producer staged an item's bitmap row and description
  B_ROWEMPTY = 25,// +buffer: its readers are done with it (8 compute warps + 2 issuers)
  B_DPAIR = 27,   // +quarter: the two warps of a row exchanged their halves of D (2 arrivals)
  B_QSFULL = 31,  // the next item's Q and dO tiles landed in shared memory (TMA)
  B_QSEMPTY = 32, // the compute warps have copied them into TMEM (8 arrivals)
  B_COUNT = 33
};
static_assert(8 * B_COUNT + 8 <= 512, "dQ kernel barrier area");

// This lane's row of a 128-row tile staged by TMA with the 128-byte swizzle (boxes of 64
// columns), this warp's half of the columns, as bf16 pairs in w; free of bank conflicts.
template <int D>
__device__ __forceinline__ void staged_row(uint32_t tile, int r, int hf, uint32_t (&w)[D / 4]) {
  constexpr int NC = D / 16;                       // 16-byte chunks in half a row
  const uint32_t box = tile + (D == 128 ? hf * 16384u : 0u);
  const int c0 = D == 128 ? 0 : hf * NC;           // first chunk of the half within the box row
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint32_t addr = swz128_chunk(box, r, c0 + c);
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[4 * c]), "=r"(w[4 * c + 1]), "=r"(w[4 * c + 2]), "=r"(w[4 * c + 3])
                 : "r"(addr));
  }
}

// This lane's half of D = sum_c dO[c] * O[c] (fp32) over the columns in w (dO) and u (O).
template <int N>
__device__ __forceinline__ float half_dot(const uint32_t (&w)[N], const uint32_t (&u)[N]) {
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < N; ++e) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[e]));
    acc = fma2(a, b, acc);
  }
  return acc.x + acc.y;
}

template <int D, int MAXNI>
__global__ void __launch_bounds__(kThreads, 1)
attn_dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
               const __grid_constant__ DqParams p) {
  using L = Smem<D>;
  constexpr int kHalf = D / 2;  // dQ columns per compute warp
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  int* const queue = p.status + 2 + 2 * (p.NT + 1) + 4;  // work queue (mask.cuh)
  if ((sbase & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment (see Smem)
    if (threadIdx.x == 0) set_status(p.status, kDevBadMeta, 0x3ff);
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
    mbar_init(bar(B_QDO), kComputeWarps);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SREAD + s), kComputeWarps);
      mbar_init(bar(B_DPFULL + s), 1);
      mbar_init(bar(B_DSFULL + s), kComputeWarps);
      mbar_init(bar(B_ROWFULL + s), 1);
      mbar_init(bar(B_ROWEMPTY + s), kComputeWarps + 2);
    }
    mbar_init(bar(B_DONE), 2);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN + 1), 1);
    mbar_init(bar(B_DQFREE), kComputeWarps);
    for (int s = 0; s < 4; ++s) mbar_init(bar(B_DPAIR + s), 2);
    mbar_init(bar(B_QSFULL), 1);
    mbar_init(bar(B_QSEMPTY), kComputeWarps);
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
  // asynchronous work issued so far, for the abort path: K and V slots and Q/dO stagings armed
  // (producer), any MMA issued (issuers)
  int gk_armed = 0, gv_armed = 0, qs_armed = 0;
  bool mma_issued = false;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
    }
    bool ok = true;
    int gbase = 0;
    for (int k = 0; ok; ++k) {
      const int rb = k & 1;
      // the row buffer is free once its readers are done with item k - 2
      if (k >= 2) {
        const bool free_ = wait(bar(B_ROWEMPTY + rb), ((k >> 1) - 1) & 1, 0x300);
        __syncwarp();
        if (!free_) { ok = false; break; }
      }
      // the next work item from the queue (schedule order: longest rows first); the end
      // marker stops every role
      int j = 0;
      if (lane == 0) j = atomicAdd(queue, 1);
      j = __shfl_sync(0xFFFFFFFFu, j, 0);
      if (j >= n_items) {
        if (lane == 0) {
          info[rb] = make_int4(-1, 0, 0, 1);
          mbar_arrive(bar(B_ROWFULL + rb));
        }
        break;
      }
      int item_idx, h;  // head-grouped chunks of the schedule (L2 locality, longest rows first)
      cta_work(j, n_items / p.H, p.H, item_idx, h);
      const int item = p.sched[item_idx];
      const int b = item >> 16, qt = item & 0xFFFF;
      const bool valid = b >= 0 && b < p.B && qt < p.NT;
      uint32_t* row = reinterpret_cast<uint32_t*>(smem + L::kRow + rb * 256u);
      int cnt = 0;
      if (valid) {
        const uint32_t* src = p.bm + (static_cast<size_t>(b) * p.NT + qt) * p.W;
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
        // Q and dO of this item into the staging tiles once the compute warps have copied the
        // previous item's into TMEM; O and the LSE, which they read from global memory, into L2
        if (qs_armed > 0 && !wait(bar(B_QSEMPTY), (qs_armed - 1) & 1, 0x309)) ok = false;
        if (ok) {
          ++qs_armed;
          mbar_arrive_expect_tx(bar(B_QSFULL), 2u * L::kTileBytes);
          for (int x = 0; x < D / 64; ++x) {
            tma_load_2d(sbase + L::kQS + x * 16384u, &tmQ, x * 64, row0 + qt * 128, bar(B_QSFULL));
            tma_load_2d(sbase + L::kdOS + x * 16384u, &tmdO, x * 64, row0 + qt * 128, bar(B_QSFULL));
          }
          const size_t r0 = static_cast<size_t>(row0) + qt * 128;
          prefetch_l2_bulk(p.o + r0 * D, L::kTileBytes);
          prefetch_l2_bulk(p.lse + r0, 512u);
        }
        int kt = next_tile(row, p.NT, 0);
        for (int n = 0; ok && n < cnt; ++n, kt = next_tile(row, p.NT, kt + 1)) {
          const int g = gbase + n, sk = g % kKStages, sv = g % kVStages;
          if (g >= kKStages && !wait(bar(B_KEMPTY + sk), ((g / kKStages) - 1) & 1, 0x301)) {
            ok = false;
            break;
          }
          gk_armed = g + 1;
          mbar_arrive_expect_tx(bar(B_KFULL + sk), L::kTileBytes);
          for (int x = 0; x < D / 64; ++x)
            tma_load_2d(sbase + L::kK + sk * L::kTileBytes + x * 16384u, &tmK, x * 64,
                        row0 + kt * 128, bar(B_KFULL + sk));
          if (g >= kVStages && !wait(bar(B_VEMPTY + sv), ((g / kVStages) - 1) & 1, 0x302)) {
            ok = false;
            break;
          }
          gv_armed = g + 1;
          mbar_arrive_expect_tx(bar(B_VFULL + sv), L::kTileBytes);
          for (int x = 0; x < D / 64; ++x)
            tma_load_2d(sbase + L::kV + sv * L::kTileBytes + x * 16384u, &tmV, x * 64,
                        row0 + kt * 128, bar(B_VFULL + sv));
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      gbase += cnt;
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ---------------------------------------------------------------- MMA issuers
    const int par = warp - kMmaWarp;  // this thread's key tiles: g % 2 == par, buffer X(par)
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc_bf16(128, 128, 0, 0);  // S = Q K^T, dP = dO V^T
      constexpr uint32_t idQ = make_idesc_bf16(128, D, 0, 1);    // dQ += dS K
      int gbase = 0, kq = 0;  // key tiles and computed items before the current one
      auto issue_s = [&](int g) -> bool {  // S(g) into X(g % 2)
        const int sk = g % kKStages;
        if (!wait(bar(B_KFULL + sk), (g / kKStages) & 1, 0x303)) return false;
        tc_fence_after();
        mma_issued = true;
        const uint32_t dK = sdesc_lo(sbase + L::kK + sk * L::kTileBytes, 16u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ts_lo(tmem + kColX + (g & 1) * 128, tmem + kColQ + 8 * kk, dK + kstep_kmajor(kk), idS,
                     kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL + (g & 1)));
        return true;
      };
      auto issue_dp = [&](int g) -> bool {  // dP(g) into X(g % 2), once S(g) has been read
        const int sv = g % kVStages;
        if (!wait(bar(B_SREAD + (g & 1)), (g >> 1) & 1, 0x306)) return false;
        if (!wait(bar(B_VFULL + sv), (g / kVStages) & 1, 0x304)) return false;
        tc_fence_after();
        const uint32_t dV = sdesc_lo(sbase + L::kV + sv * L::kTileBytes, 16u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ts_lo(tmem + kColX + (g & 1) * 128, tmem + kColDO + 8 * kk, dV + kstep_kmajor(kk),
                     idS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_DPFULL + (g & 1)));
        umma_commit(bar(B_VEMPTY + sv));
        return true;
      };
      // dQ += dS(g) K(g): dS pairs of keys [0,64) at X columns [0,32), [64,128) at [64,96).
      // Within an item, dQ(g-1) was issued by the other thread: dQ(g) waits until it has
      // completed (its K slot's release), so the accumulations never overlap; that barrier cannot
      // run a phase ahead of this wait (dQ(g+2) needs dQ(g+1), which needs dQ(g)).  The first dQ
      // of an item overwrites the accumulator once the compute warps have read the previous one.
      auto issue_dq = [&](int g, int n) -> bool {
        if (!wait(bar(B_DSFULL + (g & 1)), (g >> 1) & 1, 0x307)) return false;
        if (n >= 1) {
          if (!wait(bar(B_KEMPTY + (g - 1) % kKStages), ((g - 1) / kKStages) & 1, 0x30a))
            return false;
        } else if (kq >= 1 && !wait(bar(B_DQFREE), (kq - 1) & 1, 0x30b)) {
          return false;
        }
        tc_fence_after();
        const int sk = g % kKStages;
        const uint32_t dK = sdesc_lo(sbase + L::kK + sk * L::kTileBytes, 16384u);
        const uint32_t sX = tmem + kColX + (g & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_lo(tmem + kColDQ, sX + 64 * (kk >> 2) + 8 * (kk & 3), dK + kstep_mnmajor(kk), idQ,
                     (n > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(B_KEMPTY + sk));
        return true;
      };
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int rb = k & 1;
        if (!wait(bar(B_ROWFULL + rb), (k >> 1) & 1, 0x305)) break;
        if (info[rb].w) break;  // no more work items
        const int nt = info[rb].z;
        mbar_arrive(bar(B_ROWEMPTY + rb));
        if (nt == 0) continue;
        ok = wait(bar(B_QDO), kq & 1, 0x308);
        if (ok) tc_fence_after();
        // own tiles in order: S(g), dP(g) once S(g) is read, dQ(g) once dS(g) is written; S(g+2)
        // reuses X(par) after dQ(g) read it (tcgen05 MMAs of one thread run in issue order)
        for (int n = (par - gbase) & 1; ok && n < nt; n += 2) {
          const int g = gbase + n;
          ok = issue_s(g) && issue_dp(g) && issue_dq(g, n);
        }
        if (ok) umma_commit(bar(B_DONE));
        gbase += nt;
        ++kq;
      }
    }
  } else {
    // ---------------------------------------------------------------- compute warps 0-7
    const int quarter = warp & 3;
    const int hf = warp >> 2;           // column half of the key tile, and of dQ
    const int r = quarter * 32 + lane;  // query row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float2 scale2 = make_float2(p.scale_log2, p.scale_log2);
    bool ok = true;
    int gbase = 0, kq = 0;
    // An item's description, this row's intervals and constants are fetched one item ahead, and
    // its Q and dO are stored into TMEM before the previous item's epilogue, so that the issuers
    // can start on it while this warp writes the previous dQ.
    struct Item {
      int4 it;
      RowIntervals<MAXNI> ri;
      float lse2, negd;  // -LSE * log2(e) (-inf for a row that sees nothing) and -D, per row
      float dpart;       // this warp's half of D, until the exchange with the other half completes
      int dphase;        // phase of that exchange
    };
    int nprep = 0;  // items with key tiles prepared so far (phase of the D exchange)
    auto fetch = [&](int kf, Item& x) -> bool {
      const bool ready = wait(bar(B_ROWFULL + (kf & 1)), (kf >> 1) & 1, 0x310);
      __syncwarp();
      if (!ready) return false;
      x.it = info[kf & 1];
      if (x.it.x < 0) return true;
      const int b = x.it.x >> 16, qt = x.it.x & 0xFFFF;
      const size_t row = static_cast<size_t>(b * p.H + x.it.y) * p.S + qt * 128 + r;
      load_row_intervals(p.itab, b, p.NI, p.S, qt * 128 + r, x.ri);
      if (x.it.z == 0) return true;  // a query tile that sees no key: nothing to prepare
      const float l = p.lse[row];
      // this warp's half of the row of O (for D), from global memory (the producer prefetched it
      // into L2); then Q and dO from the staging tiles into TMEM.  The previous item's S and dP
      // MMAs, which read Q and dO in TMEM, are done: this warp has read the last dP of that item.
      constexpr int NC = D / 16;
      uint32_t u[4 * NC], w[4 * NC];
      load_rows_coalesced<NC>(u, reinterpret_cast<const char*>(p.o + (row - lane) * D + hf * (D / 2)),
                              D * 2u, lane);
      const bool staged = wait(bar(B_QSFULL), nprep & 1, 0x315);
      __syncwarp();
      if (!staged) return false;
      staged_row<D>(sbase + L::kQS, r, hf, w);
      if constexpr (D == 128) tmem_st32(tmem + lane_off + kColQ + hf * (D / 4), w);
      else tmem_st16(tmem + lane_off + kColQ + hf * (D / 4), w);
      staged_row<D>(sbase + L::kdOS, r, hf, w);
      if constexpr (D == 128) tmem_st32(tmem + lane_off + kColDO + hf * (D / 4), w);
      else tmem_st16(tmem + lane_off + kColDO + hf * (D / 4), w);
      const float dpart = half_dot(w, u);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QSEMPTY));  // the staging tiles are read
      if (lane == 0) mbar_arrive(bar(B_QDO));
      // D = rowsum(dO * O): this warp's half goes to shared memory for the other half's warp;
      // the exchange completes when the item starts (after the previous item's epilogue), so its
      // latency stays off the critical path.  A slot is rewritten only at the next item, after
      // the partner has read it.
      float* dslot = reinterpret_cast<float*>(smem + L::kDPart);  // [2 halves][128 rows]
      dslot[hf * 128 + r] = dpart;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DPAIR + quarter));
      x.dpart = dpart;
      x.dphase = nprep & 1;
      ++nprep;
      x.lse2 = l == -INFINITY ? -INFINITY : -l * 1.4426950408889634f;
      return true;
    };
    Item cur;
    cur.it = make_int4(-1, 0, 0, 0);
    ok = fetch(0, cur);
    for (int k = 0; ok && cur.it.w == 0; ++k) {
      const int rb = k & 1;
      const uint32_t* bmrow = reinterpret_cast<const uint32_t*>(smem + L::kRow + rb * 256u);
      const int nt = cur.it.z;
      const int b = cur.it.x >> 16, qt = cur.it.x & 0xFFFF;
      const size_t row0 = static_cast<size_t>(b * p.H + cur.it.y) * p.S;
      const int i = qt * 128 + r;
      if (nt > 0) {
        // the other half of D; then the per-row constants, for the dK/dV kernel that runs after
        // this one
        const float* dslot = reinterpret_cast<const float*>(smem + L::kDPart);
        const bool paired = wait(bar(B_DPAIR + quarter), cur.dphase, 0x314);
        __syncwarp();
        if (!paired) { ok = false; break; }
        const float dsum = hf == 0 ? cur.dpart + dslot[128 + r] : dslot[r] + cur.dpart;
        cur.negd = -dsum;
        if (hf == 0) {
          p.delta[row0 + i] = cur.negd;
          p.lse2[row0 + i] = cur.lse2;
        }
      }
      const float2 lse2x2 = make_float2(cur.lse2, cur.lse2), negd2 = make_float2(cur.negd, cur.negd);
      int kt = next_tile(bmrow, p.NT, 0);
      for (int n = 0; n < nt; ++n, kt = next_tile(bmrow, p.NT, kt + 1)) {
        const int g = gbase + n, xb = g & 1;
        const uint32_t sX = tmem + lane_off + kColX + xb * 128 + 64 * hf;
        bool ready = wait(bar(B_SFULL + xb), (g >> 1) & 1, 0x311);
        __syncwarp();
        if (!ready) { ok = false; break; }
        tc_fence_after();
        float pf[64];
        {
          uint32_t t0[32], t1[32];
          tmem_ld32(sX, t0);
          tmem_ld32(sX + 32, t1);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            pf[c] = __uint_as_float(t0[c]);
            pf[32 + c] = __uint_as_float(t1[c]);
          }
        }
        // S is in registers: dP may now overwrite these columns
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SREAD + xb));
        if (!tile_is_full(bmrow, kt)) {
          const int j0 = kt * 128 + 64 * hf;
          mask_cols_any(pf, j0, cur.ri, p.NI, p.check, p.masked != 0);
        }
        // P = exp2(s * scale*log2e - LSE*log2e); masked scores are -inf and give 0
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 x = fma2(make_float2(pf[c], pf[c + 1]), scale2, lse2x2);
          pf[c] = ex2_approx(x.x);
          pf[c + 1] = ex2_approx(x.y);
        }
        ready = wait(bar(B_DPFULL + xb), (g >> 1) & 1, 0x312);
        __syncwarp();
        if (!ready) { ok = false; break; }
        tc_fence_after();
        uint32_t pk[32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t dpr[32];
          tmem_ld32(sX + 32 * ch, dpr);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 gg = add2(make_float2(__uint_as_float(dpr[c]), __uint_as_float(dpr[c + 1])), negd2);
            const float2 ds = mul2(make_float2(pf[32 * ch + c], pf[32 * ch + c + 1]), gg);
            pk[16 * ch + c / 2] = pack_bf16x2(ds.x, ds.y);
          }
        }
        // dS over the columns this warp has read: keys [64*hf, +64) -> columns [64*hf, +32)
        tmem_st32(sX, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_DSFULL + xb));
      }
      // the bitmap row and the item description are no longer needed
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ROWEMPTY + rb));
      if (!ok) break;
      // the next item: description, intervals, constants, and its Q and dO into TMEM
      const Item done_item = cur;
      if (!fetch(k + 1, cur)) { ok = false; break; }  // (the producer stages an end marker last)
      if (done_item.it.x < 0) continue;  // an invalid schedule entry: nothing to write
      __nv_bfloat16* qrow = p.dq + (row0 + i) * D + hf * kHalf;
      if (nt == 0) {  // a query tile that sees no key
        uint4* dst = reinterpret_cast<uint4*>(qrow);
        for (int q = 0; q < kHalf / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
        continue;
      }
      // ---- epilogue: dQ = scale * accumulator -> bf16, this warp's half of the head dim ----
      const bool fin = wait(bar(B_DONE), kq & 1, 0x313);
      __syncwarp();
      if (!fin) { ok = false; break; }
      tc_fence_after();
      const float sc = p.scale;
      uint32_t ob[kHalf / 2];  // this row's dQ columns as bf16 pairs
#pragma unroll
      for (int c = 0; c < kHalf; c += 32) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_off + kColDQ + hf * kHalf + c, a);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          ob[(c + e) / 2] = pack_bf16x2(__uint_as_float(a[e]) * sc, __uint_as_float(a[e + 1]) * sc);
      }
      // the accumulator is free for the next item
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DQFREE));
      // rows quarter*32 .. +31 of the tile, this warp's dQ columns
      store_rows_coalesced<kHalf / 8>(
          ob, reinterpret_cast<char*>(qrow - static_cast<size_t>(lane) * D), D * 2u, lane);
      gbase += nt;
      ++kq;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up.  Copies and MMAs already issued still land in shared memory and TMEM:
    // wait for them before TMEM is freed and the CTA exits.
    if (warp == kProducerWarp && lane == 0) {
      for (int g = gk_armed - kKStages; g < gk_armed; ++g)
        if (g >= 0)
          mbar_wait_drain(bar(B_KFULL + g % kKStages), (g / kKStages) & 1, p.status, 0x3f1);
      for (int g = gv_armed - kVStages; g < gv_armed; ++g)
        if (g >= 0)
          mbar_wait_drain(bar(B_VFULL + g % kVStages), (g / kVStages) & 1, p.status, 0x3f2);
      if (qs_armed > 0) mbar_wait_drain(bar(B_QSFULL), (qs_armed - 1) & 1, p.status, 0x3f4);
    }
    if ((warp == kMmaWarp || warp == kMmaWarp + 1) && lane == 0 && mma_issued) {
      umma_commit(bar(B_DRAIN + warp - kMmaWarp));
      mbar_wait_drain(bar(B_DRAIN + warp - kMmaWarp), 0, p.status, 0x3f3);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (threadIdx.x == 0) queue_finish(queue);
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace dq

template <int D, int MAXNI>
int dq_launch(dim3 grid, cudaStream_t stream, const CUtensorMap& mk, const CUtensorMap& mv,
              const CUtensorMap& mq, const CUtensorMap& mdo, const DqParams& p) {
  const uint32_t smem = dq::Smem<D>::kAlloc;
  if (cudaFuncSetAttribute(dq::attn_dq_kernel<D, MAXNI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -1;
  dq::attn_dq_kernel<D, MAXNI><<<grid, dq::kThreads, smem, stream>>>(mk, mv, mq, mdo, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_attn_dq(const DqParams& p, int d, const void* k, const void* v, cudaStream_t stream) {
  const size_t rows = static_cast<size_t>(p.B) * p.H * p.S;
  CUtensorMap mk, mv, mq, mdo;
  if (!make_bf16_tile_map(&mk, k, rows, d) || !make_bf16_tile_map(&mv, v, rows, d) ||
      !make_bf16_tile_map(&mq, p.q, rows, d) || !make_bf16_tile_map(&mdo, p.d_o, rows, d))
    return -1;
  // persistent: one CTA per SM (one fits: 226 KB of shared memory, all 512 TMEM columns)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return -1;
  const int items = p.B * p.NT * p.H;
  const dim3 grid(items < sms ? items : sms);
  // interval registers: 4 cover every visible-form workload here; 9 the largest tables
  if (d == 128) {
    if (p.NI <= 4) return dq_launch<128, 4>(grid, stream, mk, mv, mq, mdo, p);
    return dq_launch<128, 9>(grid, stream, mk, mv, mq, mdo, p);
  }
  if (p.NI <= 4) return dq_launch<64, 4>(grid, stream, mk, mv, mq, mdo, p);
  return dq_launch<64, 9>(grid, stream, mk, mv, mq, mdo, p);
}

}  // namespace cm

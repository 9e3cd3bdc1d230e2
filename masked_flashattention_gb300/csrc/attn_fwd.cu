// Descriptor-guided attention, forward (CompileMask section 3.3.2), for sm_103a.
//
// Work item: one 128-row query tile of one (sample, head).  The Tile-State Bitmap row of that
// query tile lists the key tiles to visit: empty tiles are skipped, full tiles run without any
// mask, and partial tiles check every score against the row's intervals (mask.cuh), replacing
// invisible scores with -inf before the online softmax.
//
// Persistent CTAs: one CTA per SM; its producer warp takes the next work item of the
// longest-first schedule from a work queue (an atomic counter in the descriptor's status buffer).  Barrier phases, K/V stages and S buffers run on across items (global
// tile counter g), so the next item's Q and first K/V tiles load, and its first S MMAs run, while
// the softmax warps finish the previous item's last tiles and write its O.
//
// Each 128-key tile is split into two column halves that keep separate online-softmax states:
// half h has its own running max and row sum per query row and its own output accumulator
// O_h += P_h V_h (P_h: the half's 64 keys, V_h: the matching 64 rows of V).  The two states are
// merged once per item: O = (O_0 2^(m_0 - M) + O_1 2^(m_1 - M)) / (l_0 2^(m_0 - M) +
// l_1 2^(m_1 - M)) with M = max(m_0, m_1).  So the two warps that share a query row never wait
// for each other inside the tile loop.
//
// Warp roles (352 threads):
//   warps 0-7  softmax.  Warp w serves TMEM lane quarter w % 4 (query rows 32*(w%4) ..) and
//              column half w / 4 of each S tile.  It reads its 64 scores per row from TMEM,
//              masks partial tiles, runs its half's online softmax in the log2 domain, writes P
//              (bf16 pairs) back over the S columns it has read, rescales its half's O when the
//              running max moved, and at the end of an item merges the halves and writes O and
//              the LSE.
//   warp 8     producer: per item, stages the bitmap row in shared memory (the whole warp), then
//              lane 0 loads Q and the K and V of each visited key tile into one of 3 stages (one
//              barrier for both tiles; a stage frees when its tile's PV MMAs completed).
//   warps 9-10 MMA issuers, one thread each: the thread of warp 9 + t issues the MMAs of the key
//              tiles with g % 2 == t: S(g) = Q K(g)^T (Q and K from shared memory) and, per
//              half, O_h += P_h(g) V_h(g) with P_h read from TMEM.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O_0 [256, 256+d), O_1 [384, 384+d).  P of tile g
// lives in S buffer g % 2: keys [0,64) in columns [0,32), keys [64,128) in [64,96).
// Why two issuers: a thread that issues tcgen05 MMAs stalls on every barrier wait (even on a phase
// that is already complete), and the tensor pipe holds too few queued 128 x 128 MMAs to cover
// the stall, so a single issuer leaves a gap in the pipe at each wait.  With the tiles dealt by
// parity, one thread's MMAs run while the other waits.
// Ordering: a thread issues S(g+2) into a buffer right after PV(g), which reads P(g) from that
// buffer (tcgen05 MMAs of one thread run in issue order).  PV(g) accumulates into the O_h that
// PV(g-1) of the other thread updates, so it is issued only after PV(g-1) has completed (the
// stage barrier of tile g-1): the accumulations never overlap.  The first PV of an item
// overwrites O, once the softmax warps have read the previous item's O.  Q of the next item
// loads once both issuers have issued their last S of the current item.
// The softmax warps wait for PV(g-1) (its stage's release) only when they must rescale O: the
// completion of S(g), which they wait for anyway, already covers every PV issued before it (up to
// PV(g-2)).
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
constexpr int kStages = 3;  // K and V stage ring depth

constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;  // O_h at kColO + 128 * h

// Dynamic shared memory starts on a 1024-byte boundary here (no static shared memory); the kernel
// checks it and reports a device check failure otherwise, so the layout needs no slack.
template <int D>
struct Smem {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kKV = kTileBytes;  // stage s: K at kKV + 2*s*tile, V right after it
  static constexpr uint32_t kBar = kKV + kStages * 2u * kTileBytes;
  // per item (two buffers): the bitmap row (at most 64 words, NT <= 1024) and the item's
  // description {b << 16 | q_tile (or -1 for an invalid schedule entry), head, tile count}
  static constexpr uint32_t kRow = kBar + 256u;
  static constexpr uint32_t kInfo = kRow + 2u * 256u;
  // merge exchange of the two warps of a row: [2 halves][128 rows] of (max, sum)
  static constexpr uint32_t kPair = kInfo + 32u;
  static constexpr uint32_t kTotal = kPair + 2u * 128u * 8u;
  static constexpr uint32_t kAlloc = kTotal;
};
static_assert(Smem<128>::kAlloc <= 232448, "forward shared memory exceeds 227 KB");

enum {
  B_Q = 0,        // Q tile of the item in shared memory (TMA)
  B_KVFULL = 1,   // +stage: K and V of a key tile landed (TMA, 2 tiles of bytes)
  B_KVEMPTY = 4,  // +stage: S and PV of the stage's tile have completed (also "O is up to date",
                  // and the other issuer's go-ahead for the next PV)
  B_SFULL = 7,    // +buffer
  B_PFULL = 9,    // +buffer: P of a tile in that S buffer, both halves (8 arrivals)
  B_PAIR = 11,    // +quarter: merge exchange of a warp pair (2 arrivals per item)
  B_ALLDONE = 15, // every MMA of the item has completed (one commit per issuer per item)
  B_DRAIN = 16,   // +issuer, abort path only: every MMA the issuer issued so far has completed
  B_QEMPTY = 18,  // both issuers have issued the last S MMA of the item (one commit each)
  B_OFREE = 19,   // the softmax warps have read the item's O (8 arrivals)
  B_ROWFULL = 20, // +buffer: the producer staged an item's bitmap row and description
  B_ROWEMPTY = 22,// +buffer: its readers are done with it (8 softmax warps + 2 issuers)
  B_COUNT = 24
};

template <int D, int MAXNI>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  using L = Smem<D>;
  constexpr int kHalf = D / 2;  // output columns per softmax warp in the merge
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  int* const queue = p.status + 2 + 2 * (p.NT + 1) + 0;  // work queue (mask.cuh)
  if ((sbase & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment (see Smem)
    if (threadIdx.x == 0) set_status(p.status, kDevBadMeta, 0x1ff);
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

  // ---- set-up: barriers, TMEM -------------------------------------------------------------------
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
      mbar_init(bar(B_ROWFULL + s), 1);
      mbar_init(bar(B_ROWEMPTY + s), kSoftmaxWarps + 2);
    }
    for (int s = 0; s < 4; ++s) mbar_init(bar(B_PAIR + s), 2);
    mbar_init(bar(B_ALLDONE), 2);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN + 1), 1);
    mbar_init(bar(B_QEMPTY), 2);
    mbar_init(bar(B_OFREE), kSoftmaxWarps);
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
  // asynchronous work issued so far, for the abort path: stages armed and Q loads (producer), any
  // MMA issued (issuers)
  int g_armed = 0, q_armed = 0;
  bool mma_issued = false;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    bool ok = true;
    int gbase = 0;  // key tiles of the previous items
    for (int k = 0; ok; ++k) {
      const int rb = k & 1;
      // the row buffer is free once its readers are done with item k - 2
      if (k >= 2) {
        const bool free_ = wait(bar(B_ROWEMPTY + rb), ((k >> 1) - 1) & 1, 0x100);
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
        // Q of this item once both issuers have issued the previous item's last S
        if (q_armed > 0 && !wait(bar(B_QEMPTY), (q_armed - 1) & 1, 0x101)) ok = false;
        if (ok) {
          ++q_armed;
          mbar_arrive_expect_tx(bar(B_Q), L::kTileBytes);
          for (int x = 0; x < D / 64; ++x)
            tma_load_2d(sbase + L::kQ + x * 16384u, &tmQ, x * 64, row0 + qt * 128, bar(B_Q));
        }
        int kt = next_tile(row, p.NT, 0);
        for (int n = 0; ok && n < cnt; ++n, kt = next_tile(row, p.NT, kt + 1)) {
          const int g = gbase + n, st = g % kStages;
          if (g >= kStages && !wait(bar(B_KVEMPTY + st), ((g / kStages) - 1) & 1, 0x102)) {
            ok = false;
            break;
          }
          const uint32_t sK = sbase + L::kKV + st * 2u * L::kTileBytes;
          g_armed = g + 1;
          mbar_arrive_expect_tx(bar(B_KVFULL + st), 2u * L::kTileBytes);
          for (int x = 0; x < D / 64; ++x)
            tma_load_2d(sK + x * 16384u, &tmK, x * 64, row0 + kt * 128, bar(B_KVFULL + st));
          for (int x = 0; x < D / 64; ++x)
            tma_load_2d(sK + L::kTileBytes + x * 16384u, &tmV, x * 64, row0 + kt * 128,
                        bar(B_KVFULL + st));
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      gbase += cnt;
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ---------------------------------------------------------------- MMA issuers
    const int par = warp - kMmaWarp;  // this thread's key tiles: g % 2 == par
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc_bf16(128, 128, 0, 0);  // A = Q, B = K, both K-major
      constexpr uint32_t idO = make_idesc_bf16(128, D, 0, 1);    // A = P (TMEM), B = V MN-major
      const uint32_t dQ = sdesc_lo(sbase + L::kQ, 16u);
      int gbase = 0, kq = 0;  // key tiles and computed items before the current one
      // O_h += P_h V_h for tile g (n-th of its item): keys [64h, +64) are the K-steps
      // kk = 4h .. 4h+3.  V(g) landed before S(g) was issued (same barrier as K(g)).
      auto issue_pv = [&](int g, int n) -> bool {
        const int st = g % kStages;
        // one barrier per S buffer: the softmax warps can be at most one tile ahead of this
        // wait, so a barrier never runs two phases ahead of its waiter
        if (!wait(bar(B_PFULL + (g & 1)), (g >> 1) & 1, 0x103)) return false;
        if (n == 0) {
          // the first PV of an item overwrites O: the softmax warps must have read the previous
          // item's O (which also means that every earlier PV has completed)
          if (kq >= 1 && !wait(bar(B_OFREE), (kq - 1) & 1, 0x104)) return false;
        } else {
          // PV(g-1), issued by the other thread, has completed.  Its stage barrier cannot run
          // a phase ahead of this wait: PV(g+2) of that stage needs PV(g+1), which needs PV(g).
          if (!wait(bar(B_KVEMPTY + (g - 1) % kStages), ((g - 1) / kStages) & 1, 0x104))
            return false;
        }
        tc_fence_after();
        const uint32_t dV = sdesc_lo(sbase + L::kKV + st * 2u * L::kTileBytes + L::kTileBytes, 16384u);
        const uint32_t sP = tmem + kColS + (g & 1) * 128;
        const uint32_t acc0 = n > 0 ? 1u : 0u;
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
      // S(g) into buffer g % 2 = Q K(g)^T
      auto issue_s = [&](int g) -> bool {
        const int st = g % kStages;
        if (!wait(bar(B_KVFULL + st), (g / kStages) & 1, 0x105)) return false;
        tc_fence_after();
        mma_issued = true;
        const uint32_t dK = sdesc_lo(sbase + L::kKV + st * 2u * L::kTileBytes, 16u);
        const uint32_t dS = tmem + kColS + (g & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_lo(dS, dQ + kstep_kmajor(kk), dK + kstep_kmajor(kk), idS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL + (g & 1)));
        return true;
      };
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int rb = k & 1;
        if (!wait(bar(B_ROWFULL + rb), (k >> 1) & 1, 0x106)) break;
        if (info[rb].w) break;  // no more work items
        const int nt = info[rb].z;
        mbar_arrive(bar(B_ROWEMPTY + rb));
        if (nt == 0) continue;
        // this thread's first tile of the item, and its last S
        const int n0 = (par - gbase) & 1;
        ok = wait(bar(B_Q), kq & 1, 0x107);
        if (ok && n0 < nt) ok = issue_s(gbase + n0);
        if (ok && n0 + 2 >= nt) umma_commit(bar(B_QEMPTY));  // no further S in this item
        // per own tile: PV(n) once P(n) is written and PV(n-1) is done, and S(n+2) into the
        // buffer PV(n) reads, right behind it
        for (int n = n0; ok && n < nt; n += 2) {
          ok = issue_pv(gbase + n, n);
          if (ok && n + 2 < nt) {
            ok = issue_s(gbase + n + 2);
            if (ok && n + 4 >= nt) umma_commit(bar(B_QEMPTY));  // the last S of the item
          }
        }
        if (ok) umma_commit(bar(B_ALLDONE));
        gbase += nt;
        ++kq;
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax warps 0-7
    const int quarter = warp & 3;
    const int hf = warp >> 2;           // column half of S (keys) = index of this warp's O
    const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t my_o = tmem + lane_off + kColO + 128 * hf;
    const float sl2 = p.scale_log2;
    float2* pair_slot = reinterpret_cast<float2*>(smem + L::kPair);  // [2 halves][128 rows]
    bool ok = true;
    int gbase = 0, kq = 0;
    // An item's description and this row's intervals are fetched one item ahead, so that the
    // global loads of the intervals overlap the previous item's epilogue.
    int4 it = make_int4(-1, 0, 0, 0);
    RowIntervals<MAXNI> ri;
    auto fetch = [&](int kf, int4& itf, RowIntervals<MAXNI>& rif) -> bool {
      const bool ready = wait(bar(B_ROWFULL + (kf & 1)), (kf >> 1) & 1, 0x108);
      __syncwarp();
      if (!ready) return false;
      itf = info[kf & 1];
      if (itf.x >= 0)
        load_row_intervals(p.itab, itf.x >> 16, p.NI, p.S, (itf.x & 0xFFFF) * 128 + r, rif);
      return true;
    };
    ok = fetch(0, it, ri);
    for (int k = 0; ok && it.w == 0; ++k) {
      const int rb = k & 1;
      const uint32_t* bmrow = reinterpret_cast<const uint32_t*>(smem + L::kRow + rb * 256u);
      const int nt = it.z;
      const int b = it.x >> 16, qt = it.x & 0xFFFF, h = it.y;
      const int bh = b * p.H + h;
      const int i = qt * 128 + r;
      float m_run = -INFINITY;  // this half's running max (log2 domain)
      float l_run = 0.f;        // this half's running row sum
      int kt = next_tile(bmrow, p.NT, 0);
      for (int n = 0; n < nt; ++n, kt = next_tile(bmrow, p.NT, kt + 1)) {
        const int g = gbase + n, sb = g & 1;
        const bool s_ready = wait(bar(B_SFULL + sb), (g >> 1) & 1, 0x109);
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
        for (int q = 0; q < 21; ++q) a[q] = max3f(s[3 * q], s[3 * q + 1], s[3 * q + 2]);
        a[21] = s[63];
#pragma unroll
        for (int q = 0; q < 7; ++q) c8[q] = max3f(a[3 * q], a[3 * q + 1], a[3 * q + 2]);
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
          // rescale this half's O: PV(g-1) must be complete (PV(g-2) and earlier are, since S(g)
          // is).  Its stage barrier is at most one phase ahead of this wait: PV(g+2) needs this
          // warp's P(g+2).
          const bool o_ready =
              wait(bar(B_KVEMPTY + (g - 1) % kStages), ((g - 1) / kStages) & 1, 0x10a);
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
      // the bitmap row and the item description are no longer needed
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ROWEMPTY + rb));
      if (!ok) break;
      // the next item's description and intervals
      int4 it_next = make_int4(-1, 0, 0, 0);
      RowIntervals<MAXNI> ri_next;
      if (!fetch(k + 1, it_next, ri_next)) {  // (the producer stages an end marker last)
        ok = false;
        break;
      }
      const int4 it_cur = it;
      it = it_next;
      ri = ri_next;
      if (it_cur.x < 0) continue;  // an invalid schedule entry: nothing to write (status is set)
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.S + i) * D + hf * kHalf;
      if (nt == 0) {  // a query tile that sees no key
        uint4* dst = reinterpret_cast<uint4*>(orow);
        for (int q = 0; q < kHalf / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
        if (hf == 0) p.lse[static_cast<size_t>(bh) * p.S + i] = -INFINITY;
        continue;
      }

      // ---- epilogue: merge the two halves, O -> bf16, LSE (natural log) ----
      const bool o_final = wait(bar(B_ALLDONE), kq & 1, 0x10b);
      __syncwarp();
      if (!o_final) { ok = false; break; }
      // exchange (max, sum) with the warp of the other half
      pair_slot[hf * 128 + r] = make_float2(m_run, l_run);
      __syncwarp();
      const uint32_t pb = bar(B_PAIR + quarter);
      if (lane == 0) mbar_arrive(pb);
      const bool paired = wait(pb, kq & 1, 0x10c);
      __syncwarp();
      if (!paired) { ok = false; break; }
      const float2 ot = pair_slot[(hf ^ 1) * 128 + r];
      const float m_other = ot.x, l_other = ot.y;
      const float M = fmaxf(m_run, m_other);
      const float a_self = m_run == -INFINITY ? 0.f : ex2_approx(m_run - M);
      const float a_other = m_other == -INFINITY ? 0.f : ex2_approx(m_other - M);
      const float l_tot = l_run * a_self + l_other * a_other;
      tc_fence_after();
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const float w0 = (hf == 0 ? a_self : a_other) * inv_l;  // weight of O_0
      const float w1 = (hf == 0 ? a_other : a_self) * inv_l;  // weight of O_1
      uint32_t ob[kHalf / 2];  // this row's output columns as bf16 pairs
#pragma unroll
      for (int c = 0; c < kHalf; c += 32) {
        uint32_t o0[32], o1[32];
        tmem_ld32(tmem + lane_off + kColO + hf * kHalf + c, o0);
        tmem_ld32(tmem + lane_off + kColO + 128 + hf * kHalf + c, o1);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          ob[(c + e) / 2] = pack_bf16x2(__uint_as_float(o0[e]) * w0 + __uint_as_float(o1[e]) * w1,
                                        __uint_as_float(o0[e + 1]) * w0 + __uint_as_float(o1[e + 1]) * w1);
      }
      // O and the exchange slots are free for the next item
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OFREE));
      // rows quarter*32 .. +31 of the tile, this warp's output columns
      store_rows_coalesced<kHalf / 8>(
          ob, reinterpret_cast<char*>(orow - static_cast<size_t>(lane) * D), D * 2u, lane);
      if (hf == 0)
        p.lse[static_cast<size_t>(bh) * p.S + i] =
            l_tot > 0.f ? (M + __log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
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
      if (q_armed > 0) mbar_wait_drain(bar(B_Q), (q_armed - 1) & 1, p.status, 0x1f0);
      for (int g = g_armed - kStages; g < g_armed; ++g)
        if (g >= 0)
          mbar_wait_drain(bar(B_KVFULL + g % kStages), (g / kStages) & 1, p.status, 0x1f1);
    }
    if ((warp == kMmaWarp || warp == kMmaWarp + 1) && lane == 0 && mma_issued) {
      umma_commit(bar(B_DRAIN + warp - kMmaWarp));
      mbar_wait_drain(bar(B_DRAIN + warp - kMmaWarp), 0, p.status, 0x1f2);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (threadIdx.x == 0) queue_finish(queue);
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace fwd

template <int D, int MAXNI>
int fwd_launch(dim3 grid, cudaStream_t stream, const CUtensorMap& mq, const CUtensorMap& mk,
               const CUtensorMap& mv, const FwdParams& p) {
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
  // persistent: one CTA per SM (one fits: 227 KB of shared memory, all 512 TMEM columns)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return -1;
  const int items = p.B * p.NT * p.H;
  const dim3 grid(items < sms ? items : sms);
  // interval registers: 4 cover every visible-form workload here; 9 the largest tables
  if (d == 128) {
    if (p.NI <= 4) return fwd_launch<128, 4>(grid, stream, mq, mk, mv, p);
    return fwd_launch<128, 9>(grid, stream, mq, mk, mv, p);
  }
  if (p.NI <= 4) return fwd_launch<64, 4>(grid, stream, mq, mk, mv, p);
  return fwd_launch<64, 9>(grid, stream, mq, mk, mv, p);
}

}  // namespace cm

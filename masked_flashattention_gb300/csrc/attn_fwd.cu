// Descriptor-guided attention, forward (CompileMask section 3.3.2), for sm_103a.
//
// One CTA computes one 128-row query tile of one (sample, head).  The Tile-State Bitmap row of
// that query tile lists the key tiles to visit: empty tiles are skipped, full tiles run without
// any mask, and partial tiles check every score against the row's visible intervals with one
// unsigned subtraction and one comparison per interval (section 4.4), replacing invisible scores
// with -inf before the online softmax.
//
// Warp roles (320 threads):
//   warps 0-7  softmax.  Warp w serves TMEM lane quarter w % 4 (query rows 32*(w%4) ..) and
//              column half w / 4 of each 128-key S tile, so every query row is handled by a pair
//              of warps that exchange their partial row maxima through shared memory.  They read
//              S from TMEM, mask partial tiles, run the online softmax in the log2 domain, write
//              P (bf16 pairs) back over the S columns they have read, rescale O in TMEM when the
//              running max moved, and finally normalise O and write O and the LSE.
//   warp 8     TMA producer: Q once, then K and V of each visited key tile through two 3-slot
//              rings (a K slot frees when its S MMA completes, a V slot when its PV completes).
//   warp 9     MMA issuer (one thread): S = Q K^T and O += P V, both with the A operand (Q, P)
//              read from TMEM and the B operand (K, V) from shared memory, so shared memory
//              carries only K and V.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256+d), Q [448, 448+d/2).  P of tile n
// lives in S buffer n % 2: keys [0,64) in columns [0,32), keys [64,128) in [64,96).
// Ordering without extra barriers: the MMA issues S(n+2) into a buffer only after it saw P(n) and
// issued PV(n), which reads P(n) from that buffer; tcgen05 MMAs of one thread run in issue order.
// The softmax warps wait for PV(n-1) only when they must rescale O: the completion of S(n), which
// they wait for anyway, already covers every PV issued before it, i.e. up to PV(n-2).
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
constexpr int kMaxTiles = 1024;  // S <= 131072

constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kColQ = 448;

template <int D>
struct Smem {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kStages * kTileBytes;
  // Q is staged in K slot 2 (first needed by the third key tile, after Q has moved into TMEM)
  static constexpr uint32_t kQ = kK + 2 * kTileBytes;
  static constexpr uint32_t kRed = kV + kStages * kTileBytes;  // float [2][2][128]
  static constexpr uint32_t kBar = kRed + 2048u;
  static constexpr uint32_t kList = kBar + 256u;
  static constexpr uint32_t kTotal = kList + 2u * kMaxTiles;
  static constexpr uint32_t kAlloc = kTotal + 1024u;  // slack for 1024-byte alignment
};

enum {
  B_Q = 0,        // Q tile in shared memory (TMA)
  B_QT = 1,       // Q copied into TMEM (8 softmax warps)
  B_KFULL = 2,    // +stage
  B_VFULL = 5,    // +stage
  B_KEMPTY = 8,   // +stage: the S MMA that read the K slot has completed
  B_VEMPTY = 11,  // +stage: the PV MMA that read the V slot has completed
  B_SFULL = 14,   // +buffer
  B_PFULL = 18,   // P in TMEM and O rescaled (8 arrivals)
  B_ODONE = 19,
  B_PAIR = 20,    // +2*quarter+parity: row-max / row-sum exchange of a warp pair (2 arrivals)
  B_COUNT = 28
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  using L = Smem<D>;
  constexpr int kHalf = D / 2;  // O columns per softmax warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * B_COUNT + 4);
  int* s_ntiles = reinterpret_cast<int*>(smem + L::kBar + 8 * B_COUNT + 8);
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int item = p.sched[blockIdx.x / p.H];
  const int h = blockIdx.x % p.H;
  const int b = item >> 16;
  const int qt = item & 0xFFFF;
  const int bh = b * p.H + h;

  // ---- set-up: barriers, tile list, TMEM ----------------------------------------------------
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_Q), 1);
    mbar_init(bar(B_QT), kSoftmaxWarps);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
    }
    mbar_init(bar(B_PFULL), kSoftmaxWarps);
    mbar_init(bar(B_ODONE), 1);
    for (int s = 0; s < 8; ++s) mbar_init(bar(B_PAIR + s), 2);
    fence_barrier_init();
  }
  if (warp == 0) {
    const uint32_t* row = p.bm + (static_cast<size_t>(b) * p.NT + qt) * p.W;
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
      for (int n = 0; n < nt; ++n) {
        const int st = n % kStages;
        if (n >= kStages &&
            !mbar_wait(bar(B_KEMPTY + st), ((n / kStages) - 1) & 1, abort_flag, p.status, 0x101))
          break;
        // K slot 2 holds Q until the softmax warps have copied it into TMEM
        if (n == 2 && !mbar_wait(bar(B_QT), 0, abort_flag, p.status, 0x10c)) break;
        const int kt = list[n] & 0x3FFF;
        mbar_arrive_expect_tx(bar(B_KFULL + st), L::kTileBytes);
        for (int x = 0; x < D / 64; ++x)
          tma_load_2d(sbase + L::kK + st * L::kTileBytes + x * 16384u, &tmK, x * 64,
                      row0 + kt * 128, bar(B_KFULL + st));
        if (n >= kStages &&
            !mbar_wait(bar(B_VEMPTY + st), ((n / kStages) - 1) & 1, abort_flag, p.status, 0x10d))
          break;
        mbar_arrive_expect_tx(bar(B_VFULL + st), L::kTileBytes);
        for (int x = 0; x < D / 64; ++x)
          tma_load_2d(sbase + L::kV + st * L::kTileBytes + x * 16384u, &tmV, x * 64,
                      row0 + kt * 128, bar(B_VFULL + st));
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idS = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idO = make_idesc_bf16(128, D, 0, 1);
      bool ok = mbar_wait(bar(B_QT), 0, abort_flag, p.status, 0x102);
      auto issue_pv = [&](int m) -> bool {
        const int st = m % kStages;
        if (!mbar_wait(bar(B_PFULL), m & 1, abort_flag, p.status, 0x103)) return false;
        if (!mbar_wait(bar(B_VFULL + st), (m / kStages) & 1, abort_flag, p.status, 0x104))
          return false;
        tc_fence_after();
        const uint32_t sV = sbase + L::kV + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + kColO, tmem + kColS + (m & 1) * 128 + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                  sdesc_mnmajor(sV, kk, 16384u), idO,
                  (m > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(B_ODONE));
        umma_commit(bar(B_VEMPTY + st));
        return true;
      };
      for (int n = 0; ok && n < nt; ++n) {
        const int st = n % kStages;
        const int sb = n & 1;
        if (!mbar_wait(bar(B_KFULL + st), (n / kStages) & 1, abort_flag, p.status, 0x105)) break;
        tc_fence_after();
        const uint32_t sK = sbase + L::kK + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ts(tmem + kColS + sb * 128, tmem + kColQ + kk * 8, sdesc_kmajor(sK, kk, 16384u),
                  idS, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL + sb));
        umma_commit(bar(B_KEMPTY + st));
        if (n >= 1) ok = issue_pv(n - 1);
      }
      if (ok) issue_pv(nt - 1);
    }
  } else {
    // ---------------------------------------------------------------- softmax warps 0-7
    const int quarter = warp & 3;
    const int hf = warp >> 2;           // column half of S (keys) and of O (head dim)
    const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
    const int i = qt * 128 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // exchange slot k (k-th use) of this warp pair: write own value, meet the partner, read its
    auto pair_exchange = [&](int k, float mine, float* other) -> bool {
      float* slot = red + (k & 1) * 256;
      slot[hf * 128 + r] = mine;
      __syncwarp();
      const uint32_t pb = bar(B_PAIR + 2 * quarter + (k & 1));
      if (lane == 0) mbar_arrive(pb);
      const bool got = mbar_wait(pb, (k >> 1) & 1, abort_flag, p.status, 0x10b);
      __syncwarp();
      if (got) *other = slot[(hf ^ 1) * 128 + r];
      return got;
    };
    int st[4];
    uint32_t len[4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      st[n] = 0;
      len[n] = 0;
      if (n < p.NI) {
        const int2 iv = reinterpret_cast<const int2*>(p.itab)[(static_cast<size_t>(b) * p.NI + n) * p.S + i];
        st[n] = iv.x;
        len[n] = static_cast<uint32_t>(iv.y - iv.x);
      }
    }
    bool ok = nt > 0;
    // Q (this warp's half of the row) -> TMEM as bf16 pairs, the A operand of S = Q K^T
    const bool q_ready = ok && mbar_wait(bar(B_Q), 0, abort_flag, p.status, 0x10a);
    __syncwarp();
    if (q_ready) {
      if (D == 128) {
        uint32_t qv[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = ld_shared_v4(sbase + L::kQ + hf * 16384u + r * 128u + ((c ^ (r & 7)) << 4));
          qv[4 * c] = v.x; qv[4 * c + 1] = v.y; qv[4 * c + 2] = v.z; qv[4 * c + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + kColQ + 32 * hf, qv);
      } else {
        uint32_t qv[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t chunk = static_cast<uint32_t>(4 * hf + c);
          const uint4 v = ld_shared_v4(sbase + L::kQ + r * 128u + ((chunk ^ (r & 7)) << 4));
          qv[4 * c] = v.x; qv[4 * c + 1] = v.y; qv[4 * c + 2] = v.z; qv[4 * c + 3] = v.w;
        }
        tmem_st16(tmem + lane_off + kColQ + 16 * hf, qv);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QT));
    } else {
      ok = false;
    }

    float m_run = -INFINITY;
    float l_half = 0.f;
    const float sl2 = p.scale_log2;
    for (int n = 0; ok && n < nt; ++n) {
      const int sb = n & 1;
      const bool s_ready = mbar_wait(bar(B_SFULL + sb), (n >> 1) & 1, abort_flag, p.status, 0x107);
      __syncwarp();
      if (!s_ready) { ok = false; break; }
      tc_fence_after();
      float s[64];
      {
        uint32_t t0[32], t1[32];
        tmem_ld32(tmem + lane_off + kColS + sb * 128 + 64 * hf, t0);
        tmem_ld32(tmem + lane_off + kColS + sb * 128 + 64 * hf + 32, t1);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(t0[c]);
          s[32 + c] = __uint_as_float(t1[c]);
        }
      }

      const int entry = list[n];
      if (!(entry & 0x8000)) {
        const int j0 = (entry & 0x3FFF) * 128 + 64 * hf;
        switch (p.NI) {
          case 1: mask_cols<1>(s, j0, st, len); break;
          case 2: mask_cols<2>(s, j0, st, len); break;
          case 3: mask_cols<3>(s, j0, st, len); break;
          default: mask_cols<4>(s, j0, st, len); break;
        }
      }
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[32], s[33]);
#pragma unroll
      for (int c = 2; c < 32; c += 2) {
        mx0 = max3f(mx0, s[c], s[c + 1]);
        mx1 = max3f(mx1, s[32 + c], s[33 + c]);
      }
      float mx = fmaxf(mx0, mx1);
      // combine with the partner warp (the other column half of the same rows)
      float mx_other;
      if (!pair_exchange(n, mx, &mx_other)) { ok = false; break; }
      mx = fmaxf(mx, mx_other);
      const float m_tile = mx * sl2;
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
      l_half = l_half * alpha + ((lsa.x + lsa.y) + (lsb.x + lsb.y));

      if (n >= 1 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        // rescale O: PV(n-1) must be complete (PV(n-2) and earlier are, since S(n) is)
        const bool o_ready = mbar_wait(bar(B_ODONE), (n - 1) & 1, abort_flag, p.status, 0x108);
        __syncwarp();
        if (!o_ready) { ok = false; break; }
        tc_fence_after();
        {
#pragma unroll
          for (int c = 0; c < kHalf; c += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + kColO + hf * kHalf + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st32(tmem + lane_off + kColO + hf * kHalf + c, o);
          }
        }
      }
      // P over the S columns this warp has read: keys [64*hf, +64) -> columns [64*hf, +32)
      tmem_st32(tmem + lane_off + kColS + sb * 128 + 64 * hf, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
    }

    // ---- epilogue: O / l -> bf16, LSE (natural log) ----
    __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.S + i) * D + hf * kHalf;
    float l_tot = 0.f;
    float l_other = 0.f;
    bool o_final = ok && mbar_wait(bar(B_ODONE), (nt - 1) & 1, abort_flag, p.status, 0x109);
    __syncwarp();
    if (o_final) o_final = pair_exchange(nt, l_half, &l_other);
    if (o_final) {
      l_tot = l_half + l_other;
      tc_fence_after();
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll
      for (int c = 0; c < kHalf; c += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + kColO + hf * kHalf + c, o);
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
          l_tot > 0.f ? (m_run + __log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace fwd

int launch_attn_fwd(const FwdParams& p, int d, const void* q, const void* k, const void* v,
                    cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const uint64_t rows = static_cast<uint64_t>(p.B) * p.H * p.S;
  if (!make_bf16_tile_map(&mq, q, rows, d) || !make_bf16_tile_map(&mk, k, rows, d) ||
      !make_bf16_tile_map(&mv, v, rows, d))
    return -1;
  const dim3 grid(p.B * p.NT * p.H);
  if (d == 128) {
    const uint32_t smem = fwd::Smem<128>::kAlloc;
    if (cudaFuncSetAttribute(fwd::attn_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return -1;
    fwd::attn_fwd_kernel<128><<<grid, fwd::kThreads, smem, stream>>>(mq, mk, mv, p);
  } else {
    const uint32_t smem = fwd::Smem<64>::kAlloc;
    if (cudaFuncSetAttribute(fwd::attn_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return -1;
    fwd::attn_fwd_kernel<64><<<grid, fwd::kThreads, smem, stream>>>(mq, mk, mv, p);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace cm

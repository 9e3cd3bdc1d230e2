// Inline-PTX building blocks for sm_103a: mbarriers, TMA tile loads, tcgen05 (UMMA) with
// TMEM accumulators, and the shared-memory / instruction descriptors those MMAs consume.
//
// Layout convention used by every kernel in this library: a 128-row tile of 16-bit elements is
// stored as one or more "boxes" of 64 columns (128 bytes) x 128 rows, each box 16 KB and
// 1024-byte aligned, written by TMA with the 128-byte swizzle (16-byte chunk c of row r lands at
// chunk c ^ (r % 8)).  The same bytes can be handed to the tensor core in two ways:
//   * K-major: rows are the M (or N) index, the 64 columns are K.  Atoms of 8 rows x 128 B are
//     SBO = 1024 B apart; a K step of 16 elements moves the start address by 32 B inside a box.
//   * MN-major: rows are K, the 64 columns are M (or N).  The next 64 M/N columns live in the next
//     box (LBO = 16 KB); 8-row K groups are SBO = 1024 B apart; a K step of 16 rows is +2048 B.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace cm {

// ----------------------------------------------------------------------------------------------
// status word: kernels never trap; a bounded wait that gives up records a code and returns.
// ----------------------------------------------------------------------------------------------
enum : int {
  kDevOk = 0,
  kDevTimeout = 1,      // an mbarrier wait exceeded its limit
  kDevBadMeta = 2,      // segment metadata not monotone / not ending at S
  kDevDescMismatch = 3, // backward Tile-State Bitmap is not the transposed forward bitmap
  kDevBadSchedule = 4,  // a schedule entry names no tile row of the descriptor
};

__device__ __forceinline__ void set_status(int* status, int code, int where) {
  if (status != nullptr) atomicCAS(status, 0, (code << 16) | (where & 0xFFFF));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ----------------------------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded waits.  Every wait of a role on a phase that another role completes goes through
// WaitCtl: it gives up after `limit_ns` (a kernel parameter; 2 s unless the host lowered it), sets
// the CTA's `abort` flag (shared memory) and the status word, and returns false.  Once the flag is
// set, every later WaitCtl wait of the CTA returns false at once, so all roles leave their loops
// quickly.  Before the CTA frees TMEM and exits, the roles that issued asynchronous work (TMA
// copies, tcgen05 MMAs) wait for it with mbar_wait_drain: that work completes by itself, whatever
// the other roles did, so these waits end; they are bounded all the same.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr uint64_t kDrainLimitNs = 2000000000ull;

struct WaitCtl {
  volatile int* abort;
  int* status;
  uint64_t limit_ns;
  __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity, int where) const {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (mbar_try_wait(bar, parity)) return true;
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        set_status(status, kDevTimeout, where);
        return false;
      }
    }
  }
};

// Wait for a phase whose completion needs no other role (copies or MMAs already issued by the
// calling thread), ignoring the abort flag.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, int* status,
                                                int where) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDrainLimitNs) {
      set_status(status, kDevTimeout, where);
      return false;
    }
  }
  return true;
}

// ----------------------------------------------------------------------------------------------
// TMA
// ----------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
// Hint: bring `bytes` (a multiple of 16) at `ptr` into L2.  Skipped for an address that is not
// 16-byte aligned (the bulk prefetch requires it).
__device__ __forceinline__ void prefetch_l2_bulk(const void* ptr, uint32_t bytes) {
  if ((reinterpret_cast<uint64_t>(ptr) & 15u) != 0) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(ptr)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// store of a shared-memory tile (laid out as a TMA load of the same box would leave it) into
// global memory through a tensor map; completion is tracked with bulk groups of the issuing thread
__device__ __forceinline__ void tma_store_2d(const void* tmap, int32_t x, int32_t y, uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until no committed bulk group of this thread still reads shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// wait until every committed bulk group of this thread has completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// make generic-proxy shared-memory writes visible to the async proxy (tensor core / TMA)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads / stores
// ----------------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]  (kind::f16: both operands bf16 here, fp32 accumulate)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on `bar` once every previously issued tcgen05 op of this thread has completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// instruction descriptor, kind::f16, bf16 x bf16 -> f32, dense
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, int a_mn_major,
                                                       int b_mn_major) {
  return (1u << 4)                                // D format f32
         | (1u << 7)                              // A format bf16
         | (1u << 10)                             // B format bf16
         | (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// shared-memory matrix descriptor with the 128-byte swizzle
__host__ __device__ constexpr uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                        uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) |
         (static_cast<uint64_t>(1) << 46)  // descriptor version for tcgen05
         | (static_cast<uint64_t>(2) << 61);  // 128-byte swizzle
}
// K-major operand, 16-element K step `kk` of a tile made of 64-column boxes `box_bytes` apart
__device__ __forceinline__ uint64_t sdesc_kmajor(uint32_t tile, int kk, uint32_t box_bytes) {
  const uint32_t addr = tile + static_cast<uint32_t>(kk >> 2) * box_bytes +
                        static_cast<uint32_t>(kk & 3) * 32u;
  return make_sdesc_sw128(addr, 16u, 1024u);
}
// MN-major operand (rows = K), 16-row K step `kk`; the 64-wide MN blocks are boxes apart
__device__ __forceinline__ uint64_t sdesc_mnmajor(uint32_t tile, int kk, uint32_t box_bytes) {
  const uint32_t addr = tile + static_cast<uint32_t>(kk) * 2048u;
  return make_sdesc_sw128(addr, box_bytes, 1024u);
}

// The same SW128 descriptors split into halves for a lean issue loop.  The high word (stride
// 1024 B, version, swizzle) is one constant for every operand here; the low word holds the
// address field (bits 0-13, address >> 4) and the leading byte offset.  A shared address below
// 256 KB gives an address field below 2^14, so the K step of an operand is one 32-bit add of
// (step offset >> 4) to its base low word: no carry leaves the field.
constexpr uint32_t kSdescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__host__ __device__ constexpr uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
// low-word offset of K step kk: K-major (64-column boxes 16 KB apart, 32 B per step inside a
// box) and MN-major (16 rows of 128 B per step)
__host__ __device__ constexpr uint32_t kstep_kmajor(int kk) {
  return static_cast<uint32_t>(kk >> 2) * (16384u >> 4) + static_cast<uint32_t>(kk & 3) * 2u;
}
__host__ __device__ constexpr uint32_t kstep_mnmajor(int kk) {
  return static_cast<uint32_t>(kk) * (2048u >> 4);
}
// the split form gives the full descriptors bit for bit (last K step of a tile at 208 KB)
static_assert(make_sdesc_sw128(0x34000u + 16384u + 3 * 32u, 16u, 1024u) ==
                  ((static_cast<uint64_t>(kSdescHi) << 32) | (sdesc_lo(0x34000u, 16u) + kstep_kmajor(7))),
              "K-major split descriptor");
static_assert(make_sdesc_sw128(0x34000u + 7 * 2048u, 16384u, 1024u) ==
                  ((static_cast<uint64_t>(kSdescHi) << 32) | (sdesc_lo(0x34000u, 16384u) + kstep_mnmajor(7))),
              "MN-major split descriptor");
__device__ __forceinline__ void umma_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 da, {%1, %5};\n\t"
      "mov.b64 db, {%2, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kSdescHi)
      : "memory");
}
__device__ __forceinline__ void umma_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 db, {%2, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kSdescHi)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane (quarter*32 + t), cols c..c+31
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
// named barrier over `count` threads (ids 1..15; 0 is __syncthreads)
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------------------------------------
// coalesced row stores
// ----------------------------------------------------------------------------------------------
// A warp holds 32 consecutive rows of a tile, one per lane (lane t: row t), each as NC 16-byte
// chunks in w[4c .. 4c+3].  Read or written as they are, every memory instruction would touch 32
// rows (32 memory segments).  transpose_chunks swaps the roles of lane and chunk index within each
// group of NC lanes with three (NC = 8) or two (NC = 4) rounds of butterfly shuffles: at distance
// d, lane pairs (l, l ^ d) exchange the chunks whose index differs from their lane in bit d.  So
// "lane NC*G + t holds chunk c of row NC*G + t in w[4c..]" becomes "lane NC*G + c holds chunk c of
// row NC*G + q in w[4q..]", and back: one memory instruction then covers 32/NC whole row segments
// of NC * 16 bytes.
template <int NC>
__device__ __forceinline__ void transpose_chunks(uint32_t (&w)[4 * NC], int lane) {
  static_assert(NC == 4 || NC == 8, "chunks per row segment");
#pragma unroll
  for (int d = 1; d < NC; d <<= 1) {
    const bool up = (lane & d) != 0;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      if (j & d) continue;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t x = up ? w[4 * j + e] : w[4 * (j | d) + e];
        const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, d);
        if (up) {
          w[4 * j + e] = y;
        } else {
          w[4 * (j | d) + e] = y;
        }
      }
    }
  }
}
// Stores the warp's 32 rows; `base` is the address of row 0's first chunk for this warp.
template <int NC>
__device__ __forceinline__ void store_rows_coalesced(uint32_t (&w)[4 * NC], char* base,
                                                     size_t row_stride, int lane) {
  transpose_chunks<NC>(w, lane);
  const int c = lane % NC, g0 = lane - c;  // chunk of this lane, first row of its group
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    uint4* dst = reinterpret_cast<uint4*>(base + static_cast<size_t>(g0 + q) * row_stride) + c;
    *dst = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}
// Loads the warp's 32 rows (lane t gets row t) with the same coalesced pattern.
template <int NC>
__device__ __forceinline__ void load_rows_coalesced(uint32_t (&w)[4 * NC], const char* base,
                                                    size_t row_stride, int lane) {
  const int c = lane % NC, g0 = lane - c;
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    const uint4 v = *(reinterpret_cast<const uint4*>(base + static_cast<size_t>(g0 + q) * row_stride) + c);
    w[4 * q] = v.x;
    w[4 * q + 1] = v.y;
    w[4 * q + 2] = v.z;
    w[4 * q + 3] = v.w;
  }
  transpose_chunks<NC>(w, lane);
}

// ----------------------------------------------------------------------------------------------
// small numeric helpers
// ----------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// paired fp32 arithmetic (one instruction for two lanes of data): d = a * b + c, a + b, a * b.
// The compiler's own paired-float builtins, so that it places the operand pairs in registers
// itself (no moves into and out of 64-bit pairs around each instruction).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
// three-input maximum
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// pack two floats into a bf16x2 word (round to nearest even); `lo` goes to the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Address of the 16-byte chunk c of row r in a box of 128-byte rows laid out with the 128-byte
// swizzle (what a TMA load of the box with that swizzle leaves in shared memory, and what a TMA
// store of it expects; the box starts on a 1024-byte boundary): r * 128 + ((c ^ (r % 8)) * 16).
// The 8 lanes of a quarter-warp that access the same chunk of 8 consecutive rows hit 8 different
// 16-byte bank groups.
__device__ __forceinline__ uint32_t swz128_chunk(uint32_t box, int r, int c) {
  return box + static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(c) ^ (r & 7)) << 4);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace cm

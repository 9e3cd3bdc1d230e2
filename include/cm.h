/*
 * cm.h -- C ABI of the descriptor-guided masked attention library (libcm.so).
 *
 * The operations follow "CompileMask: Bridging the Gap Between Expressiveness and Efficiency in
 * Attention Masking":
 *   - section 3.2 (MaskSpec, Regions with a row guard and a visibility rule) and section 3.2.2
 *     (symbolic lowering: AST, DNF normalisation, interval extraction, canonicalisation)
 *       -> cm_compile_spec / cm_spec_* (offline, host only);
 *   - section 3.3 and 3.3.1 (online preprocess kernel evaluating the compiled endpoints against
 *     batch metadata; Execution Descriptor = Interval Table padded with zero-length intervals
 *     plus 2-bit Tile-State Bitmaps; separate forward and backward descriptors)
 *       -> cm_descriptor_sizes / cm_build_descriptor;
 *   - section 3.3.2 (descriptor-guided attention: skip empty tiles, run full tiles unmasked,
 *     check partial tiles against the endpoints with unsigned arithmetic, -inf before the
 *     online softmax) and section 4.4 (unsigned visible-interval check)
 *       -> cm_attn_fwd / cm_attn_bwd.
 *
 * Conventions shared by every entry point
 *   - Every pointer named "device" must point to memory of the current CUDA device.  The library
 *     allocates no device memory: the caller owns every buffer and must keep it alive until the
 *     work queued on `stream` has finished.  The only heap object the library owns is the host
 *     cm_spec returned by cm_compile_spec (free it with cm_spec_free).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device work is queued on it and
 *     the call returns without waiting; nothing runs on the CPU in place of a kernel.
 *   - Return value: CM_OK (0) or a negative CM_ERR_* code.  Arguments are validated on the host
 *     before anything is queued; a call that fails validation queues nothing.  Errors detected on
 *     the device (bad segment metadata, a bounded wait that expired) are recorded in the
 *     descriptor's status word and reported by cm_get_status.
 *   - Tensors Q, K, V, O, dO, dQ, dK, dV are bf16, contiguous, layout [B][H][S][d].  The LSE is
 *     fp32 [B][H][S] in natural log.  Row i of a descriptor is a query row (forward) or a key
 *     column (backward).
 *   - Supported shapes: d in {64, 128}; S a positive multiple of 128; tile = 128; at most 2^24
 *     heads (CM_ERR_UNSUPPORTED above that).
 */
#ifndef CM_H_
#define CM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CM_API __attribute__((visibility("default")))

enum {
  CM_OK = 0,
  CM_ERR_PARSE = -1,        /* spec text does not parse or uses an unsupported form */
  CM_ERR_INVALID_ARG = -2,  /* null pointer, bad size, descriptor/shape mismatch */
  CM_ERR_UNSUPPORTED = -3,  /* valid request outside the supported shapes (d, S, tile, limits) */
  CM_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed */
  CM_ERR_TIMEOUT = -5,      /* device status: a bounded wait inside a kernel expired */
  CM_ERR_DEVICE_CHECK = -6, /* device status: segment metadata failed validation */
  CM_ERR_DESC_MISMATCH = -7 /* device status: the backward descriptor's Tile-State Bitmap is not
                               the transpose of the forward one (the two MaskSpecs do not
                               describe the same mask) */
};

/* Opaque compiled MaskSpec (host memory, owned by the caller after cm_compile_spec). */
typedef struct cm_spec cm_spec;

/* Per-batch metadata (section 1 / 2.2: sequence lengths and segment boundaries).
 *   seg  device int32 [B][nseg_max + 1]: seg[b][0] = 0, strictly increasing up to
 *        seg[b][nseg[b]] = S; entries after nseg[b] are ignored.
 *   nseg device int32 [B]: segment count of each sample, 1 <= nseg[b] <= nseg_max. */
typedef struct cm_meta {
  const int32_t* seg;
  const int32_t* nseg;
  int32_t nseg_max;
} cm_meta;

/* Execution Descriptor (section 3.3.1), forward and backward halves.  All buffers are device
 * memory allocated by the caller with the sizes from cm_descriptor_sizes.
 *   form    CM_FORM_VISIBLE (the paper's representation): the Interval Tables hold each row's
 *           visible intervals, ni_f / ni_b = the specs' interval counts.  CM_FORM_MASKED (the
 *           representation section 4.4 compares it with): they hold the maximal runs of
 *           invisible indices of each row in increasing order, ni_f / ni_b = the specs' counts
 *           + 1.  The bitmaps and schedules are the same in both forms.
 *   itab_f  int32 [B][ni_f][S][2]  (start, end) of each visible key interval of query row i,
 *           half open; unused slots and empty intervals are (0, 0)
 *   bm_f    uint32 [B][S/tile][ceil((S/tile)/16)]  2 bits per (q-tile, k-tile):
 *           0 empty, 1 partial, 2 full; k-tile t at bits 2*(t % 16) of word t / 16
 *   itab_b  int32 [B][ni_b][S][2]  visible query intervals of key column j
 *   bm_b    uint32 [B][S/tile][ceil((S/tile)/16)]  (k-tile, q-tile) states
 *   sched_f int32 [B * S/tile]  forward work order: (b << 16 | q_tile), most tiles first
 *   sched_b int32 [B * S/tile]  backward work order: (b << 16 | k_tile), most tiles first
 *   status  int32 [2 + 2 * (S/tile + 1) + 6]  device error word (first element), then the
 *           preprocess kernel's grid barrier and schedule histograms, then the work queues of
 *           the three attention kernels (a next-item counter and a finished-CTA counter each,
 *           returned to zero by the last CTA of every launch); cleared by cm_build_descriptor.
 *           Attention calls that use one descriptor must therefore run one after another (one
 *           stream, or ordered by events), never at the same time. */
#define CM_FORM_VISIBLE 0
#define CM_FORM_MASKED 1
typedef struct cm_descriptor {
  int32_t B, S, tile, ni_f, ni_b, form;
  int32_t* itab_f;
  uint32_t* bm_f;
  int32_t* itab_b;
  uint32_t* bm_b;
  int32_t* sched_f;
  int32_t* sched_b;
  int32_t* status;
} cm_descriptor;

/* ---- offline compiler (host only; section 3.2.2) ------------------------------------------- */

/* Parse and lower a MaskSpec.  Text: one Region per line,
 *     region <guard> : <rule>
 * <guard> is `all` or a boolean expression of the row index i; <rule> is a boolean expression
 * over i and the other index j (&&, ||, !, comparisons < <= > >= == !=).  Integer terms: i, j,
 * S, nseg, integer constants, + - and multiplication by a constant, % by a positive constant
 * (non-negative remainder), min(a, b), max(a, b),
 * seg_idx(e), seg_start(e), seg_end(e), seg_start_at(k), seg_end_at(k).  Lines starting with '#'
 * are comments.  Regions are tried in order; the first whose guard holds applies to the row.
 * On success *out receives a new cm_spec.  On CM_ERR_PARSE a message is written to err (if
 * err_len > 0). */
CM_API int cm_compile_spec(const char* text, cm_spec** out, char* err, size_t err_len);

/* Free a spec from cm_compile_spec (NULL is ignored). */
CM_API void cm_spec_free(cm_spec* spec);

/* The compiler-derived interval count (max slots over the Regions), section 3.3.1. */
CM_API int cm_spec_num_intervals(const cm_spec* spec, int* ni_max);

/* Human-readable lowered form (Regions, slot endpoints, slot conditions) written to buf as a
 * NUL-terminated string; *needed (if not NULL) receives the full length + 1.  Host only. */
CM_API int cm_spec_describe(const cm_spec* spec, char* buf, size_t len, size_t* needed);

/* CUDA C++ source of the mask-specific preprocess kernel (section 3.1: the compiler generates a
 * mask-specific preprocess kernel) of a (forward, backward) pair of specs: their two row
 * evaluators and the shared kernel body "descriptor_core.cuh", which the library carries in
 * itself; one launch of it builds both halves of the descriptor and both schedules.  Written to
 * buf as a NUL-terminated string; *needed (if not NULL) receives the full length + 1.  Host
 * only. */
CM_API int cm_descriptor_kernel_source(const cm_spec* fwd, const cm_spec* bwd, char* buf,
                                       size_t len, size_t* needed);

/* Whether the pair's generated kernel can run.  load = 0: compile it with NVRTC only (host only,
 * no GPU needed).  load = 1: compile it and load it into the current device context, which is
 * what cm_build_descriptor does on its first call with the pair (the result, good or bad, is kept
 * with the forward spec; compiling takes a few tenths of a second).  Returns CM_OK on success,
 * CM_ERR_UNSUPPORTED when NVRTC (libnvrtc.so.13) cannot be opened, CM_ERR_CUDA when compiling or
 * loading failed.  The NVRTC log or the failing step goes to log as a NUL-terminated string (log
 * may be NULL). */
CM_API int cm_descriptor_kernel_status(const cm_spec* fwd, const cm_spec* bwd, int load, char* log,
                                       size_t log_len);

/* cm_descriptor_kernel_source / _status with `spec` as both the forward and the backward spec
 * (one spec's generated code on its own). */
CM_API int cm_spec_kernel_source(const cm_spec* spec, char* buf, size_t len, size_t* needed);
CM_API int cm_spec_kernel_status(const cm_spec* spec, int load, char* log, size_t log_len);

/* ---- online descriptor construction (sections 3.3, 3.3.1) ---------------------------------- */

/* Byte sizes of the descriptor buffers, in the order itab_f, bm_f, itab_b, bm_b, sched_f,
 * sched_b, status, for the given form (CM_FORM_VISIBLE or CM_FORM_MASKED).  tile must be 128.
 * Use the status size as given: the status word may be followed by counters of the preprocess
 * kernel. */
CM_API int cm_descriptor_sizes(const cm_spec* fwd, const cm_spec* bwd, int B, int S, int tile,
                               int form, size_t sizes[7]);

/* Which descriptor kernel cm_build_descriptor runs, for the whole process:
 * CM_PREPROCESS_GENERATED (default): the generated kernel of the (forward, backward) spec pair;
 *   if it cannot be compiled or loaded (see cm_descriptor_kernel_status), the generic kernel runs
 *   instead;
 * CM_PREPROCESS_GENERIC: the generic kernel, which interprets the compiled endpoint programs.
 * Either way one cooperative launch builds both halves and both schedules.
 * Both are GPU kernels and build identical descriptors.  Returns CM_ERR_INVALID_ARG for any other
 * mode.  Not synchronised with builds in flight on other host threads. */
#define CM_PREPROCESS_GENERATED 0
#define CM_PREPROCESS_GENERIC 1
CM_API int cm_set_preprocess_mode(int mode);

/* Queue the preprocess kernel that evaluates both specs against `meta` and fills `desc`: a
 * memset of desc->status (the status word and the kernel's counters), then one cooperative
 * launch (all its blocks resident at once; they meet at one grid barrier before the schedules
 * are written).  desc->B, S, tile, form, ni_f, ni_b must match the specs and sizes; its
 * pointers must be set.  Asynchronous on `stream`. */
CM_API int cm_build_descriptor(const cm_spec* fwd, const cm_spec* bwd, const cm_meta* meta,
                               int B, int S, cm_descriptor* desc, void* stream);

/* ---- descriptor-guided attention (section 3.3.2) -------------------------------------------- */

/* Form of the attention kernels' partial-tile check, for the whole process (full and empty
 * tiles never run one; the forms of section 4.4's ablation plus the default):
 * CM_CHECK_UNSIGNED: per score, for each stored interval [s, e) one subtraction and one unsigned
 *   comparison, (uint32)(x - s) < (uint32)(e - s) (the paper's test);
 * CM_CHECK_TWO_COMPARE: per score, s <= x && x < e for each stored interval;
 * CM_CHECK_RANGE_MASK (default): per row and 32 indices, each stored interval becomes a range
 *   of bits of a 32-bit mask (clamped unsigned differences), and each score tests one bit.
 * With a CM_FORM_MASKED descriptor an index is visible iff it lies in none of the stored
 * intervals.  All forms give the same results.  Returns CM_ERR_INVALID_ARG for any other mode.
 * Not synchronised with launches in flight on other host threads. */
#define CM_CHECK_UNSIGNED 0
#define CM_CHECK_TWO_COMPARE 1
#define CM_CHECK_RANGE_MASK 3
CM_API int cm_set_interval_check(int mode);

/* Forward: o = softmax(scale * q k^T masked by desc) v; lse = natural-log row sums.
 * q, k, v, o: device bf16 [B][H][S][d]; lse: device fp32 [B][H][S].  The mask is shared by
 * all heads of a sample.  A row with no visible key gets o = 0 and lse = -inf. */
CM_API int cm_attn_fwd(const cm_descriptor* desc, const void* q, const void* k, const void* v,
                       void* o, float* lse, int B, int H, int S, int d, float scale,
                       void* stream);

/* Workspace bytes cm_attn_bwd needs: per-row D = rowsum(dO * O) and LSE * log2(e), fp32 (8 bytes
 * per row of B*H*S, each array rounded up to 256 bytes). */
CM_API int cm_attn_bwd_workspace_size(int B, int H, int S, int d, size_t* bytes);

/* Backward: dq, dk, dv (device bf16 [B][H][S][d]) of sum(o * dO) given the forward's o and lse.
 * Section 3.3: each traversal direction has its own descriptor.  Two kernels, the stages below
 * in this order: dQ along query tiles with the forward half of the descriptor (itab_f, bm_f,
 * sched_f), which also writes D and LSE * log2(e) into the workspace, then dK and dV along key
 * tiles with the backward half (itab_b, bm_b, sched_b), which read them.  Every output element is written exactly
 * once (no atomics), so results are deterministic.  `workspace` (device, >= the size above,
 * 16-byte aligned) is overwritten.  Every argument is checked before the first stage is queued.
 * The dK/dV stage also checks on the device that bm_b is the transpose of bm_f and records
 * CM_ERR_DESC_MISMATCH in the status word when it is not (the computation still runs). */
CM_API int cm_attn_bwd(const cm_descriptor* desc, const void* q, const void* k, const void* v,
                       const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes, int B, int H, int S,
                       int d, float scale, void* stream);

/* The stages of cm_attn_bwd, for callers that queue or time them one by one.  cm_attn_bwd queues
 * cm_attn_bwd_dq, then cm_attn_bwd_dkdv, on one stream with one workspace.
 *   cm_attn_bwd_dq        dq along query tiles with the forward descriptor; reads q, k, v, o, lse,
 *                         d_o (device, layouts as above) and writes the workspace: per row of
 *                         every query tile that sees at least one key, -D = -sum_c dO[c] * O[c]
 *                         and -LSE * log2(e) (-inf for a row that sees nothing), fp32;
 *   cm_attn_bwd_dkdv      dk, dv along key tiles with the backward descriptor (section 3.3);
 *                         reads q, k, v, d_o and the workspace written by cm_attn_bwd_dq (or by
 *                         cm_attn_bwd_prologue) earlier on the same stream;
 *   cm_attn_bwd_prologue  writes the whole workspace (every row) from o, lse and d_o alone, for
 *                         callers that run cm_attn_bwd_dkdv without cm_attn_bwd_dq.
 * Same argument rules and error codes as cm_attn_bwd. */
CM_API int cm_attn_bwd_prologue(const void* o, const float* lse, const void* d_o, void* workspace,
                                size_t workspace_bytes, int B, int H, int S, int d,
                                void* stream);
CM_API int cm_attn_bwd_dkdv(const cm_descriptor* desc, const void* q, const void* k,
                            const void* v, const void* d_o, void* dk, void* dv,
                            const void* workspace, size_t workspace_bytes, int B, int H, int S,
                            int d, float scale, void* stream);
CM_API int cm_attn_bwd_dq(const cm_descriptor* desc, const void* q, const void* k, const void* v,
                          const void* o, const float* lse, const void* d_o, void* dq,
                          void* workspace, size_t workspace_bytes, int B, int H, int S, int d,
                          float scale, void* stream);

/* Limit of every bounded wait inside the attention kernels, for the whole process, in ns
 * (0 restores the default of 2 s; at most 60 s, else CM_ERR_INVALID_ARG).  A wait that reaches it
 * makes its CTA stop: the CTA waits for the copies and MMAs it already issued, records
 * CM_ERR_TIMEOUT in the status word (cm_get_status) and exits, leaving the outputs of the work
 * items it had not finished unwritten (the call's outputs are then undefined); the context and
 * the descriptor stay usable.  This is a diagnostic hook: a very small limit makes ordinary waits
 * expire, which tests the time-out path without a fault.  Not synchronised with launches in
 * flight on other host threads.  (The pages describe no failure handling; this is the library's
 * own.) */
CM_API int cm_set_wait_limit_ns(unsigned long long ns);

/* ---- backward without a workspace (no counterpart in the paper) ---------------------------- */

/* Size of the library's built-in backward scratch array (32 MiB per GPU that loads libcm.so). */
#define CM_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Same computation and arguments as cm_attn_bwd, minus the workspace, for callers that cannot
 * allocate device memory themselves: plugins whose host framework owns all device memory, or
 * latency-critical threads that must not call cudaMalloc (it can synchronise the device).  The
 * scratch comes from a fixed file-scope device array inside the library instead, so this call
 * allocates nothing.
 *   - Limit: the workspace cm_attn_bwd_workspace_size reports must fit CM_NOALLOC_SCRATCH_BYTES
 *     (B*H*S <= 4,194,304 rows); larger problems return CM_ERR_UNSUPPORTED and queue
 *     nothing.
 *   - The array's device address is looked up (cudaGetSymbolAddress) on the first call on each
 *     device, with that device current; make that first call before any stream capture.
 *   - The array is held by every GPU that loads the library until the process exits.
 *   - All calls share the one array per device, and it keeps the previous call's contents.
 *     Each call first rewrites the part it reads (8 bytes per row of B*H*S: D and
 *     LSE * log2(e)), so nothing needs clearing.  Calls whose work overlaps on the GPU, e.g. on
 *     two streams, race on it: order them on one stream. */
CM_API int cm_attn_bwd_noalloc(const cm_descriptor* desc, const void* q, const void* k,
                               const void* v, const void* o, const float* lse, const void* d_o,
                               void* dq, void* dk, void* dv, int B, int H, int S, int d,
                               float scale, void* stream);

/* ---- status --------------------------------------------------------------------------------- */

/* Wait for `stream`, then read desc->status: CM_OK, CM_ERR_TIMEOUT, CM_ERR_DEVICE_CHECK or
 * CM_ERR_DESC_MISMATCH, the first error recorded since cm_build_descriptor cleared the word
 * (CM_ERR_CUDA if the wait or copy itself failed). */
CM_API int cm_get_status(const cm_descriptor* desc, void* stream);

/* Static description of a CM_* code. */
CM_API const char* cm_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* CM_H_ */

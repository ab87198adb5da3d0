/*
 * fa2.h — C ABI of the GB300 (sm_103a) FlashAttention-2 library: the forward
 * pass and its gradient (fa2_bwd).
 *
 * The operation (FlashAttention-2 forward):
 *   for every batch b, head h and query row i of an N-long sequence,
 *     S_ij = scale * <Q[b,h,i,:], K[b,h,j,:]>      over the allowed keys j
 *     O[b,h,i,:] = softmax_j(S_ij) V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp(S_ij)              (natural log)
 *   Allowed keys: 0 <= j < N, and j <= i when is_causal != 0 (top-left
 *   aligned, query and key sequences have the same length N).
 * Definition and the statistics kept: "FlashAttention-2 MMA 代码学习"
 * (chuoer47 blog), step 0 (O = softmax(QK^T/sqrt(d)) V) and step 1 (the
 * row-wise (m, l) merge); the yangyitao.com CUDA book, ch. 15, section 15.1
 * (LSE = m + log l is the one statistic kept for the backward pass) and
 * section 15.3 (the kernel signature Q, K, V, O, LSE, N, H, softmax_scale,
 * is_causal; scale applied before the max; causal masking of col > row;
 * padded columns >= N masked; rows >= N not written; an all-masked row
 * gives O = 0 and LSE = +inf, which the masks supported here never produce).
 *
 * All entry points are thread-safe and may be called from several host
 * threads at once.
 */
#ifndef FA2_GB300_H
#define FA2_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the same type as cudaStream_t / CUstream */

/* The library is built with hidden symbol visibility; only the entry points
 * below are exported. */
#if defined(__GNUC__)
#define FA2_API __attribute__((visibility("default")))
#else
#define FA2_API
#endif

/* dtype codes */
#define FA2_F16 0  /* IEEE binary16 inputs and output */
#define FA2_BF16 1 /* bfloat16 inputs and output      */

/* schedule codes of fa2_fwd_sched and fa2_bwd_sched */
#define FA2_SCHED_AUTO 0     /* the one with less work on the busiest SM (what fa2_bwd uses) */
#define FA2_SCHED_UNITS 1    /* whole work units dealt to the SMs in rounds */
#define FA2_SCHED_BALANCED 2 /* equal steps per SM; units cut between SMs are merged */

/* status codes (0 = success, negative = error) */
#define FA2_OK 0
#define FA2_ERR_INVALID_ARG (-1) /* null pointer, negative size, bad scale, overlapping O/LSE/inputs, size overflow */
#define FA2_ERR_UNSUPPORTED (-2) /* head dim not supported, unknown dtype, device is not sm_103 */
#define FA2_ERR_ALIGN (-3)       /* a tensor pointer is not 16-byte aligned */
#define FA2_ERR_CUDA (-4)        /* a CUDA runtime/driver call failed (see fa2_last_cuda_error) */
#define FA2_ERR_TIMEOUT (-5)     /* the device watchdog fired (returned by fa2_device_status) */

/*
 * fa2_fwd — enqueue the forward pass on `stream`.
 *
 * Q, K, V : device pointers, contiguous [B, H, N, D] tensors of `dtype`
 *           (row-major, D fastest). Read only. 16-byte aligned.
 * O       : device pointer, contiguous [B, H, N, D] of `dtype`. Fully
 *           overwritten with the normalised output, rounded to nearest-even.
 *           Must not overlap Q, K, V or LSE.
 * LSE     : device pointer, contiguous [B, H, N] fp32. Fully overwritten with
 *           the natural-log logsumexp of each row's scaled scores. 16-byte
 *           aligned; must not overlap Q, K, V or O.
 * B, H, N : batch, heads, sequence length (queries and keys), each >= 0. If
 *           any is 0 the call does nothing and returns FA2_OK (pointers may
 *           then be NULL).
 * D       : head dimension; 32, 64, 96, 128, 256, 512 or 1024. 64 and 128
 *           are the native tile widths; 32 and 96 run in the tiles of 64 and
 *           128, whose columns past D the kernel reads as zeros. These four
 *           are the head dims the split-Q launcher of "FlashAttention-2 MMA
 *           代码学习" dispatches (its host function at the end of the page).
 *           256, 512 and 1024 are the tiling_qk page's larger ones: 256 runs
 *           on a kernel of its own with 128-row work units; 512 and 1024 tile
 *           the output's head dimension, a work unit being 128 query rows and
 *           one 256-column chunk of O, each recomputing the scores over all
 *           of D (the tensor cores do 1.5x / 2.5x the FLOPs of the
 *           definition). 512 and 1024 always run the round schedule.
 * scale   : multiplier on Q.K; finite and > 0 (the usual value is 1/sqrt(D)).
 * is_causal: nonzero keeps only keys j <= i for query i.
 * dtype   : FA2_F16 or FA2_BF16.
 * stream  : CUDA stream (NULL = legacy default stream) of the current device;
 *           all pointers must be device memory of that device.
 *
 * Ownership: the caller owns every buffer; the library never allocates,
 * frees or retains them. Asynchronous: a return of FA2_OK means the kernel
 * was enqueued, not that it finished; errors inside the kernel surface as a
 * CUDA error on the stream or through fa2_device_status. Host-side argument
 * errors are detected before anything is enqueued and leave O and LSE
 * untouched.
 */
FA2_API int fa2_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
            int B, int H, int N, int D, float scale, int is_causal, int dtype,
            struct CUstream_st* stream);

/*
 * fa2_fwd_workspace_bytes — bytes of device workspace fa2_fwd_ws needs on the
 * current device for head dimension D (32, 64, 96, 128, 256, 512 or 1024):
 * one fp32 partial result of a work unit per SM (256 rows, or 128 at head
 * dim 256) plus one 8-byte flag per 128-row sub-tile; 0 at head dims 512 and
 * 1024, which run the round schedule only. It does not depend on B, H or N. Returns FA2_OK, FA2_ERR_INVALID_ARG (bytes NULL),
 * FA2_ERR_UNSUPPORTED (D) or FA2_ERR_CUDA.
 */
FA2_API int fa2_fwd_workspace_bytes(int D, size_t* bytes);

/*
 * fa2_fwd_ws — the same operation, arguments and results as fa2_fwd, with a
 * caller-owned device workspace that lets the kernel balance work exactly
 * across the SMs: each persistent CTA takes an equal share of all
 * (query tile, K/V tile) steps, and a query tile whose K/V range is cut
 * between CTAs is finished by merging fp32 partial results with the online
 * (m, l) rule of "FlashAttention-2 MMA 代码学习", step 1 (the merge the
 * pages apply across K/V blocks, here applied across CTAs). At head dims
 * 512 and 1024 it runs the round schedule of fa2_fwd (the workspace unused).
 *
 * workspace: NULL (then this is exactly fa2_fwd), or a 16-byte aligned
 *   device buffer of at least fa2_fwd_workspace_bytes(D) bytes that overlaps
 *   no tensor. Its contents need no initialisation and are scratch after the
 *   call; calls that share a workspace must not run concurrently on the GPU.
 * The launch is cooperative (all CTAs resident); if that cannot be arranged
 * the call returns FA2_ERR_CUDA.
 * Errors as fa2_fwd, plus FA2_ERR_INVALID_ARG for a workspace that is too
 * small or overlaps a tensor, FA2_ERR_ALIGN for a misaligned workspace.
 */
FA2_API int fa2_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* LSE,
               int B, int H, int N, int D, float scale, int is_causal, int dtype,
               void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * fa2_fwd_sched — the same operation, arguments and results as fa2_fwd, with
 * the work schedule chosen by the caller or by the library:
 *   FA2_SCHED_UNITS: the round schedule of fa2_fwd (whole 256-row query
 *     units, 128-row from head dim 256, dealt to persistent CTAs in rounds;
 *     heaviest first in a zig-zag when causal). `workspace` may be NULL.
 *   FA2_SCHED_BALANCED: the stream-K schedule of fa2_fwd_ws; `workspace`
 *     (as described there) is required, except at head dims 512 and 1024,
 *     which always run the round schedule and need none.
 *   FA2_SCHED_AUTO: the schedule fa2_fwd_schedule_for names for this
 *     problem on the current device; with a NULL workspace always the round
 *     schedule.
 * Both schedules compute the same function; they differ in the order of the
 * fp32 sums (outputs within rounding of each other) and each is
 * deterministic. This is the call for a C caller who wants the faster
 * schedule without choosing it: on a 152-SM GB300, B=1 H=8 N=8192 D=128
 * non-causal runs balanced (its 256 units leave 48 SMs idle in the second
 * round), B=4 H=16 N=4096 D=128 causal runs in rounds.
 * Errors as fa2_fwd_ws, plus FA2_ERR_INVALID_ARG for an unknown schedule code
 * or FA2_SCHED_BALANCED without a workspace.
 */
FA2_API int fa2_fwd_sched(const void* Q, const void* K, const void* V, void* O, float* LSE,
                  int B, int H, int N, int D, float scale, int is_causal, int dtype,
                  void* workspace, size_t workspace_bytes, int schedule, struct CUstream_st* stream);

/*
 * fa2_fwd_schedule_for — the schedule FA2_SCHED_AUTO takes for a problem on a
 * device with `sms` SMs (FA2_SCHED_UNITS or FA2_SCHED_BALANCED into
 * *schedule). The cost of each is the busiest SM's work in K/V-tile steps
 * (one query unit against one 128-key tile): the rounds take
 * ceil(units / sms) * tiles per unit; the balanced schedule takes
 * units * tiles per unit / sms, plus 4 steps for the write and merge of the
 * partial results of the units it cuts. Balanced is named when it is at
 * least 5 % cheaper, and never for causal work (the zig-zag rounds measured
 * faster there). Host arithmetic only: needs no device.
 * Returns FA2_OK, FA2_ERR_INVALID_ARG (NULL output, negative size, sms < 1)
 * or FA2_ERR_UNSUPPORTED (D).
 */
FA2_API int fa2_fwd_schedule_for(int B, int H, int N, int D, int is_causal, int sms, int* schedule);

/*
 * fa2_fwd_noalloc — the same operation, arguments and results as fa2_fwd,
 * with the balanced (stream-K) schedule of fa2_fwd_ws, for callers that
 * cannot allocate device memory: code that must not call cudaMalloc, for
 * instance because its host application owns all device memory through a
 * fixed pool or arena and allows no other allocation, or because it runs on a
 * latency-critical path where an allocation and the device synchronisation
 * it implies are not acceptable. It calls no allocation routine. The pages
 * have no counterpart to this entry point.
 *
 * Its scratch is one static device array of this library, 21,465,600 bytes,
 * held on every GPU where it has been loaded until the process exits. It
 * covers devices of up to 160 SMs at every supported head dimension; a device with
 * more SMs is refused with FA2_ERR_UNSUPPORTED.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Under lazy module loading (the default since CUDA 12) that first call is
 * also when the 21 MB are committed on the device, so it can fail with
 * FA2_ERR_CUDA (out of memory) if the caller's pool already holds nearly all
 * of it: make one warm-up call at start-up, before sizing such a pool.
 * All calls share the array and it keeps the last call's contents. Nothing
 * in it has to start at zero: each launch tags its partial results with a
 * unique value, so leftovers of earlier calls are never read. Calls that
 * overlap on the GPU (on different streams, or on different host threads
 * without ordering) race on the array and must not be made.
 * Errors as fa2_fwd.
 */
FA2_API int fa2_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    int B, int H, int N, int D, float scale, int is_causal, int dtype,
                    struct CUstream_st* stream);

/*
 * fa2_fwd_host_buffer_bytes — bytes of device staging memory fa2_fwd_host
 * needs for a [B, H, N, D] problem on the current device: room for Q, K, V,
 * O (B*H*N*D 16-bit values each), LSE (B*H*N floats plus 12 bytes of
 * alignment padding per head) and the balanced schedule's workspace, each
 * rounded up to 256 bytes. Returns FA2_OK,
 * FA2_ERR_INVALID_ARG (bytes NULL, negative size, B*H above INT32_MAX),
 * FA2_ERR_UNSUPPORTED (D) or FA2_ERR_CUDA (no usable device).
 */
FA2_API int fa2_fwd_host_buffer_bytes(int B, int H, int N, int D, size_t* bytes);

/*
 * fa2_fwd_host — the same operation and results as fa2_fwd, from and to HOST
 * memory: Q, K, V are copied to the device, the forward pass runs there and
 * O, LSE are copied back, in chunks of whole heads so that copies in both
 * directions overlap the computation of other chunks. The pages have no
 * counterpart to this entry point (their kernels take device tensors).
 *
 * Q, K, V : host pointers, contiguous [B, H, N, D] of `dtype`. Read only.
 * O, LSE  : host pointers, contiguous [B, H, N, D] of `dtype` and [B, H, N]
 *           fp32; fully overwritten. Must not overlap the inputs or each
 *           other. Page-locked memory (cudaHostAlloc / cudaHostRegister) is
 *           needed for the copies to overlap anything; pageable memory works
 *           but the copies then run one after another.
 * Copies  : each copy costs the copy engine a few microseconds besides its
 *           bytes, so the call makes as few as the layout allows. When K
 *           and V follow Q at one fixed spacing (three slices of one packed
 *           [3, B, H, N, D] buffer, for one), each chunk's Q, K and V move in
 *           one two-dimensional copy, else in three. When the device can
 *           address LSE directly (page-locked memory under unified
 *           addressing; cudaPointerGetAttributes gives its device pointer)
 *           and N is a multiple of 4, the kernels write LSE there and no LSE
 *           copy is made. Either way the results are the same.
 * B, H, N, D, scale, is_causal, dtype: as fa2_fwd.
 * heads_per_chunk: heads (of the flattened B*H) per chunk; 0 = ceil(B*H / 4).
 *           The first chunk holds half as many (rounded down, at least one)
 *           so that the first kernel starts sooner; the last holds what
 *           remains.
 * balanced: nonzero runs each chunk on the balanced schedule of fa2_fwd_ws
 *           (workspace inside dev_buffer), zero on the schedule of fa2_fwd.
 * dev_buffer, dev_bytes: caller-owned device staging memory of the current
 *           device, 256-byte aligned, at least fa2_fwd_host_buffer_bytes
 *           bytes. Its contents are scratch: they need no initialisation
 *           and are not part of the result.
 * stream  : the ordering stream (NULL = legacy default stream). The copies
 *           run on two non-blocking streams the library creates once per
 *           device and keeps until the process exits; they start after the
 *           work already queued on `stream`, and work queued on `stream`
 *           after the call starts only once every copy is complete. The host
 *           buffers must stay valid, and unmodified for Q, K, V, until then.
 *
 * Ownership: the caller owns every buffer; the library allocates no memory.
 * Asynchronous as fa2_fwd: synchronise `stream` before reading O or LSE.
 * Argument errors are detected before anything is enqueued. If a CUDA call
 * fails part way, the chunks enqueued before it still complete, `stream` is
 * still ordered behind them, and the call returns FA2_ERR_CUDA (O and LSE
 * are then partly written). Calls for one device are enqueued one at a time
 * (an internal lock); calls that share a dev_buffer must be ordered by the
 * caller.
 */
FA2_API int fa2_fwd_host(const void* Q, const void* K, const void* V, void* O, float* LSE,
                 int B, int H, int N, int D, float scale, int is_causal, int dtype,
                 int heads_per_chunk, int balanced, void* dev_buffer, size_t dev_bytes,
                 struct CUstream_st* stream);

/*
 * fa2_bwd_workspace_bytes — bytes of device workspace fa2_bwd needs for these
 * sizes: an fp32 dQ accumulator [B, H, N, D], two fp32 row statistics of
 * B*H*ceil(N/64)*64 entries each, and the balanced schedule's partial
 * results (160 slots of 2*128*D floats) and their 160 8-byte flags, every
 * part rounded up to 256 bytes.
 * Returns FA2_OK, FA2_ERR_INVALID_ARG (bytes NULL or a negative size) or
 * FA2_ERR_UNSUPPORTED (D not 32, 64, 96 or 128). Needs no device.
 */
FA2_API int fa2_bwd_workspace_bytes(int B, int H, int N, int D, size_t* bytes);

/*
 * fa2_bwd — enqueue the backward pass (the gradient of fa2_fwd's O with
 * respect to Q, K and V for an upstream gradient dO) on `stream`.
 *
 * The operation, for every (b, h), with P the softmax weights of the forward:
 *   dV = P^T dO,  dP = dO V^T,  Delta_i = <dO_i, O_i>,  dS = P * (dP - Delta)
 *   dQ = scale * dS K,  dK = scale * dS^T Q
 * P is recomputed from Q, K and LSE (P_ij = exp(S_ij - LSE_i)); S and P never
 * reach device memory; the outer loop runs over K/V tiles and dQ is summed
 * across them with fp32 atomic adds. Source: the yangyitao.com CUDA book,
 * ch. 15, section 15.1 (change 4: only LSE is kept for the backward pass)
 * and the chapter's closing paragraph (S and P recomputed, dQ accumulated
 * atomically, outer loop over K/V).
 *
 * Q, K, V : device pointers, the forward's inputs ([B, H, N, D], `dtype`).
 * O, LSE  : the forward's outputs for those inputs (fa2_fwd's O and LSE).
 * dO      : device pointer, [B, H, N, D] of `dtype`: the upstream gradient.
 * dQ, dK, dV: device pointers, [B, H, N, D] of `dtype`. Fully overwritten,
 *           rounded to nearest-even. Must not overlap each other, an input
 *           or the workspace.
 * B, H, N, D, scale, is_causal, dtype: as for fa2_fwd (the same values the
 *           forward was called with), except that D is 32, 64, 96 or 128
 *           (32 and 96 run in the tiles of 64 and 128, as in the forward).
 * workspace: device memory of at least fa2_bwd_workspace_bytes(B, H, N, D)
 *           bytes, 256-byte aligned, owned by the caller. Its contents on
 *           entry do not matter; it is scratch for the duration of the call
 *           on `stream` and must not be used by other work until the call's
 *           kernels have finished.
 * stream  : CUDA stream of the current device (NULL = legacy default).
 *
 * All tensor pointers must be 16-byte aligned. Three kernels are enqueued in
 * order (row statistics, the backward, dQ conversion). Errors as fa2_fwd,
 * plus FA2_ERR_INVALID_ARG for a missing or too small workspace and
 * FA2_ERR_ALIGN for a misaligned one. The library allocates nothing.
 */
FA2_API int fa2_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
            const float* LSE, void* dQ, void* dK, void* dV,
            int B, int H, int N, int D, float scale, int is_causal, int dtype,
            void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * fa2_bwd_sched — fa2_bwd with the work schedule of its main kernel chosen
 * by the caller (fa2_bwd is this call with FA2_SCHED_AUTO):
 *   FA2_SCHED_UNITS: each SM takes whole K/V tiles (all their query steps)
 *     in rounds; with B*H*ceil(N/128) tiles not a multiple of the SM count
 *     the last round leaves SMs idle.
 *   FA2_SCHED_BALANCED: each SM (at most 160 of them) takes an equal share
 *     of all (K/V tile, query step) pairs; a tile cut between SMs is
 *     finished by the SM holding its first steps, which adds the fp32
 *     partial dK, dV of the others (left in the workspace) before writing
 *     dK and dV. The launch is cooperative (all SMs' blocks resident); if
 *     that cannot be arranged the call returns FA2_ERR_CUDA.
 *   FA2_SCHED_AUTO: the one whose busiest SM has fewer query steps
 *     (balanced only if at least 5 % fewer).
 * The results are the same up to fp32 summation order; each schedule is
 * deterministic for dK and dV. Errors as fa2_bwd, plus FA2_ERR_INVALID_ARG
 * for an unknown schedule code.
 */
FA2_API int fa2_bwd_sched(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* LSE, void* dQ, void* dK, void* dV,
                  int B, int H, int N, int D, float scale, int is_causal, int dtype,
                  void* workspace, size_t workspace_bytes, int schedule, struct CUstream_st* stream);

/*
 * fa2_device_status — read the device-side watchdog word of the current
 * device, synchronising `stream` first. *status receives 0 when no kernel of
 * this library has timed out waiting on one of its internal barriers since
 * the last clear, else a positive code identifying the wait that gave up.
 * If `clear` is nonzero the word is reset to 0 afterwards. Returns FA2_OK
 * (no timeout), FA2_ERR_TIMEOUT (a timeout was recorded; *status holds its
 * site), FA2_ERR_INVALID_ARG (status NULL), FA2_ERR_UNSUPPORTED (not an
 * sm_103 device) or FA2_ERR_CUDA.
 */
FA2_API int fa2_device_status(struct CUstream_st* stream, int* status, int clear);

/*
 * fa2_set_watchdog_ns — set the time (in nanoseconds) a kernel waits on any
 * one internal barrier before it records a timeout in the watchdog word and
 * winds down. Applies to launches made after the call, process-wide. 0
 * restores the default (1 s). Returns FA2_OK.
 */
FA2_API int fa2_set_watchdog_ns(unsigned long long ns);

/*
 * fa2_test_withhold_next_load — test hook for the watchdog. When enable is
 * nonzero, the next launch of this library (process-wide, one launch only:
 * a forward kernel, or the main kernel of fa2_bwd) withholds its first K/V
 * tile: the waits for that tile run out after the watchdog time, the kernel
 * records the wait site in the watchdog word, winds down without leaving
 * work in flight, and its outputs (O/LSE, or dQ/dK/dV) are left unspecified.
 * No GPU fault, trap or hang is involved. Returns FA2_OK.
 */
FA2_API int fa2_test_withhold_next_load(int enable);

/* Human-readable text for a status code (static storage, never NULL). */
FA2_API const char* fa2_error_string(int code);

/* Text of the last CUDA error seen by this library on the calling thread
 * (static thread-local storage, never NULL; "" if none). */
FA2_API const char* fa2_last_cuda_error(void);

/* Library ABI version: (major << 16) | minor. */
FA2_API int fa2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA2_GB300_H */

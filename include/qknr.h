/*
 * qknr.h -- C ABI of libqknr: fused, in-place, per-head QK RMSNorm + rotary
 * position embedding (RoPE) on NVIDIA GB300 (sm_103a).
 *
 * What one call computes (fused_inplace_qknorm_rope deep-dive, §2.1-§2.3):
 * for every token t and every head h of q (weight q_w) and of k (weight k_w),
 * with x = the head's head_dim values and p = positions[t]:
 *
 *     r   = 1 / sqrt( (1/head_dim) * sum_i x_i^2 + eps )          (§2.1, §4.3)
 *     n_i = x_i * r * w_i                                          (§2.1)
 *     c_j = cache[p][j], s_j = cache[p][rope_dim/2 + j]            (§2.2, §3)
 *     interleaved (GPT-J), j < rope_dim/2:                          (§2.2)
 *         o_{2j} = n_{2j} c_j - n_{2j+1} s_j,  o_{2j+1} = n_{2j+1} c_j + n_{2j} s_j
 *     NeoX (LLaMA), d < rope_dim/2:                                 (§2.2, §4.4)
 *         o_d = n_d c_d - n_{d+R/2} s_d,       o_{d+R/2} = n_{d+R/2} c_d + n_d s_d
 *     o_i = n_i for rope_dim <= i < head_dim (partial RoPE)         (§2.2)
 *
 * and writes o back over x, rounded once to the tensor's dtype (round to
 * nearest even). All arithmetic is fp32. The tensor contract follows §3 of
 * the same page: q [T, n_qo, D] and k [T, n_kv, D] in fp16 or bf16 with unit
 * innermost stride; q_w, k_w [D] in the same dtype; cos_sin_cache fp32
 * [cache_len, rope_dim], cos in the first half of each row and sin in the
 * second; positions [T] int32 or int64. The op returns nothing and allocates
 * nothing per call.
 *
 * Thread / device model: every entry point acts on the calling thread's
 * current CUDA device. qknr_init must have been called for that device.
 * Calls are asynchronous on the given stream except where stated.
 *
 * Errors: every entry point returns a QKNR_* status. Nothing is thrown across
 * the ABI. On a non-OK status, qknr_last_error() returns a message for the
 * calling thread. A failed validation launches nothing and leaves q and k
 * untouched.
 */
#ifndef QKNR_H
#define QKNR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype argument: element type of q, k, q_w, k_w, OR-ed with the positions type */
#define QKNR_BF16 0x000    /* bfloat16 q/k/weights */
#define QKNR_FP16 0x001    /* IEEE half q/k/weights */
#define QKNR_POS_I64 0x100 /* positions are int64 (otherwise int32) */
/*
 * QKNR_INPUTS_READY, OR-ed into dtype, is the caller's promise that q_w, k_w
 * and positions were not written by the kernel enqueued just before this call
 * on the stream (for example: weights loaded at start-up, positions computed
 * at the start of the forward pass, and a GEMM producing q and k just before).
 * With it, the kernels read the weights and positions while that
 * kernel finishes (programmatic dependent launch), and read q, k and the
 * cos|sin table only after it has completed: about 17% less latency per
 * decode-sized call and 3% more bandwidth on a 4608-token DiT call, with the
 * same results. Breaking the promise is a data race. The unfused baseline and
 * the staged host path (which launches without the early start) ignore it.
 */
#define QKNR_INPUTS_READY 0x200

/* status codes */
#define QKNR_OK 0
#define QKNR_ERR_NOT_INITIALIZED 1 /* qknr_init was not called for the current device */
#define QKNR_ERR_INVALID_ARG 2     /* null pointer, negative or oversized size, overlapping q/k, bad dtype */
#define QKNR_ERR_UNSUPPORTED 3     /* head_dim / rope_dim / pairing outside the accepted set */
#define QKNR_ERR_MISALIGNED 4      /* pointer or stride breaks the 16-byte vector rule */
#define QKNR_ERR_CUDA 5            /* a CUDA runtime call failed; message has the CUDA error */
#define QKNR_ERR_POSITION_OOB 6    /* qknr_apply_checked: a position outside [0, cache_len) */

/*
 * Prepare the library for CUDA device `device`: reads the SM count and other
 * limits, and allocates a 16-byte status block (the position-check counters
 * of qknr_apply_checked).
 * Idempotent; safe to call from several threads. Restores the caller's
 * current device before returning. Returns QKNR_OK or QKNR_ERR_CUDA /
 * QKNR_ERR_INVALID_ARG (no such device).
 */
int qknr_init(int device);

/*
 * Release what qknr_init allocated, and the streams and events of the
 * host-buffer pipeline (qknr_apply_host), on every device. Callers must make
 * sure no launch from this library is still running. After it, qknr_init
 * must be called again before any apply.
 */
int qknr_shutdown(void);

/* Message for the calling thread's last non-OK status ("" if none). */
const char *qknr_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int qknr_version(void);

/*
 * Shape gate, the counterpart of the deep-dive's can_use check (§5.2) for
 * this library's own kernels. Returns 1 if (head_dim, rope_dim, is_neox,
 * dtype) is in the accepted set, else 0. Accepted: head_dim in {64, 80, 96,
 * 128, 192, 256}; rope_dim even with 0 < rope_dim <= head_dim; interleaved
 * pairing takes every such rope_dim; NeoX pairing takes rope_dim % 16 == 0 or
 * rope_dim in {2, 4, 6, 8}. This contains the page's set (head_dim/32 elements per lane,
 * rotary lanes a power of two) and more.
 */
int qknr_can_use(int head_dim, int rope_dim, int is_neox, int dtype);

/*
 * The fused op, in place, asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream).
 *
 * q, k          device pointers to head (t=0, h=0) of q and k; modified in place.
 * q_w, k_w      device pointers to the [head_dim] RMSNorm weights, q/k dtype.
 * cos_sin_cache device pointer to fp32 [cache_len, rope_dim], row-major.
 * positions     device pointer to [num_tokens] int32 or int64 (QKNR_POS_I64).
 *               A position outside the cache is undefined behaviour here, as
 *               on the page (§4.4); qknr_apply_checked checks them.
 * num_tokens    T >= 0 (0: nothing is launched).
 * n_qo, n_kv    query and key head counts, each >= 1 (GQA: n_qo != n_kv), and
 *               n_qo + n_kv <= 2^24.
 * head_dim      D; rope_dim R: see qknr_can_use.
 * is_neox       0 = interleaved (GPT-J) pairing, 1 = NeoX pairing.
 * q_stride      elements between consecutive tokens of q; k_stride the same for k.
 * head_stride   elements between consecutive heads, shared by q and k (§3).
 *               The innermost stride is 1. Heads must not overlap
 *               (head_stride >= D) and token rows must not overlap.
 * eps           added to the mean of squares inside the square root.
 * dtype         QKNR_BF16 or QKNR_FP16, OR-ed with QKNR_POS_I64 for int64 positions.
 *
 * Alignment: q, k, q_w, k_w 16-byte aligned; q_stride, k_stride, head_stride
 * multiples of 8 elements; cos_sin_cache 4-byte aligned; positions aligned to
 * their size. q and k must not overlap (disjoint views of one fused QKV buffer
 * are fine). Neither q nor k may span more than 2^56 bytes, and no size or
 * stride may exceed 2^56 (QKNR_ERR_INVALID_ARG), so that no byte offset can
 * wrap. The caller owns every buffer; nothing is retained after return.
 *
 * Kernels: the library has two kernels with identical results, chosen per
 * call by a measured rule (or by qknr_tune / qknr_set_tuning): the register
 * kernel, which loads each warp item straight into registers (decode-sized
 * calls), and the ring kernel, which double-buffers each warp's items in
 * shared memory with asynchronous copies (every larger call), in one of two
 * issue orders (QKNR_TUNE_RING_ORDER).
 */
int qknr_apply(void *q, void *k, const void *q_w, const void *k_w, const float *cos_sin_cache,
               const void *positions, int64_t num_tokens, int n_qo, int n_kv, int head_dim,
               int rope_dim, int is_neox, int64_t q_stride, int64_t k_stride, int64_t head_stride,
               float eps, int dtype, void *stream);

/*
 * qknr_apply plus a check of every position against [0, cache_len). Tokens
 * whose position is outside are left untouched; all others are computed as by
 * qknr_apply. SYNCHRONOUS: waits for `stream` before returning. Returns
 * QKNR_ERR_POSITION_OOB (message: count and first bad token) if any position
 * was out of range. Uses the status word that qknr_init allocated, so calls
 * on one device must not overlap on the GPU (they serialise on the host).
 */
int qknr_apply_checked(void *q, void *k, const void *q_w, const void *k_w,
                       const float *cos_sin_cache, int64_t cache_len, const void *positions,
                       int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim,
                       int is_neox, int64_t q_stride, int64_t k_stride, int64_t head_stride,
                       float eps, int dtype, void *stream);

/*
 * The unfused two-kernel chain that the fused op replaces, for measuring the
 * fusion benefit on this GPU (deep-dive §2.4 table, and the §6 fallback of
 * RMSNorm then RoPE): an RMSNorm kernel writes the normalised, weighted q and
 * k back in place, rounded to their dtype; a RoPE kernel then reads them
 * again, rotates the first rope_dim dims and writes them. Two launches, two
 * reads and two writes of Q and K instead of one of each. Same arguments and
 * errors as qknr_apply; asynchronous on `stream`. The intermediate rounding
 * makes results differ from qknr_apply by up to one unit in the last place
 * of each rotated pair's length.
 */
int qknr_apply_unfused(void *q, void *k, const void *q_w, const void *k_w,
                       const float *cos_sin_cache, const void *positions, int64_t num_tokens,
                       int n_qo, int n_kv, int head_dim, int rope_dim, int is_neox,
                       int64_t q_stride, int64_t k_stride, int64_t head_stride, float eps,
                       int dtype, void *stream);

/*
 * qknr_apply_checked without any allocation, for callers that cannot call
 * cudaMalloc (a runtime that owns every device allocation or a pre-sized
 * pool, a plug-in whose host reserves the allocator). The op itself has no
 * counterpart of this entry point on the deep-dive page; it exists only for
 * such callers.
 *
 * Same arguments, results and QKNR_ERR_POSITION_OOB report as
 * qknr_apply_checked, but qknr_init is not needed and nothing is allocated:
 * the 16-byte status block lives in a 256-byte file-scope __device__ array
 * of the library, which every GPU that loads the library holds until the
 * process exits. A call needs those 16 bytes whatever its num_tokens, so no
 * problem size exceeds the array. The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current.
 * No call of this entry point can be captured into a CUDA graph: each one
 * reads its status back to the host and synchronises. That set-up is kept for
 * the life of the process: a device reset (cudaDeviceReset) after the first
 * call on a device is not supported by this entry point. Each call resets
 * the status it reads, and waits for `stream` before returning (it is
 * synchronous, like qknr_apply_checked). All calls share the one array:
 * calls on one device are serialised on the host, and two launches that used
 * the array at the same time on the GPU would race.
 */
int qknr_apply_checked_noalloc(void *q, void *k, const void *q_w, const void *k_w,
                               const float *cos_sin_cache, int64_t cache_len,
                               const void *positions, int64_t num_tokens, int n_qo, int n_kv,
                               int head_dim, int rope_dim, int is_neox, int64_t q_stride,
                               int64_t k_stride, int64_t head_stride, float eps, int dtype,
                               void *stream);

/*
 * qknr_apply for q and k whose heads are laid out with different strides
 * (for example q inside a fused QKV buffer and k in a padded cache layout):
 * q's heads are q_head_stride elements apart, k's k_head_stride. The
 * deep-dive's contract (§3, §4.7) has one shared head stride; this entry
 * point lifts that restriction. Same results, bit for bit, as qknr_apply on
 * the same values. With equal strides, or one head on a side, it is
 * qknr_apply's single launch; otherwise two launches on `stream`, q's heads
 * then k's, each with the kernel the rule picks for that side. Arguments, ownership and errors as
 * qknr_apply (each side's stride is checked on its own; a negative stride is
 * QKNR_ERR_INVALID_ARG). Asynchronous on `stream`.
 */
int qknr_apply_strided(void *q, void *k, const void *q_w, const void *k_w,
                       const float *cos_sin_cache, const void *positions, int64_t num_tokens,
                       int n_qo, int n_kv, int head_dim, int rope_dim, int is_neox,
                       int64_t q_stride, int64_t k_stride, int64_t q_head_stride,
                       int64_t k_head_stride, float eps, int dtype, void *stream);

/* qknr_apply_host flags */
#define QKNR_HOST_AUTO 0   /* direct when every host buffer is device-mapped, else staged */
#define QKNR_HOST_STAGED 1 /* always copy through the device staging buffers */
#define QKNR_HOST_DIRECT 2 /* always direct; QKNR_ERR_INVALID_ARG if a buffer is not device-mapped */

/*
 * The op on q, k and positions held in HOST memory, for callers whose
 * activations live on the host (offload, or a host-side pipeline): the
 * results are written back into h_q and h_k. Same operation and results as
 * qknr_apply (deep-dive §3 contract); the host transfer is this library's
 * addition.
 *
 * h_q, h_k, h_positions: host buffers, laid out by the same sizes and strides
 *   as for qknr_apply. Only the heads' bytes are read and written: bytes
 *   between heads and between rows (the V part of a fused QKV buffer) are
 *   left as they are.
 * q_w, k_w, cos_sin_cache: device memory, as for qknr_apply.
 * d_q, d_k, d_positions: caller-owned device buffers with the same layout,
 *   used only by the staged mode (may be NULL when the call runs direct).
 *
 * Direct mode: when the host buffers are pinned memory mapped into the
 * device's address space (cudaHostAlloc, cudaHostRegister, torch's
 * pin_memory on a unified-addressing system) or managed memory, checked with
 * cudaPointerGetAttributes at both ends of each buffer, one kernel reads and
 * writes them in place over the host link (NVLink-C2C on GB300), both
 * directions at once.
 * Staged mode: the tokens are cut into chunks of chunk_tokens (0: automatic,
 *   up to 8 chunks of at least 4 MB); chunk i is copied into the staging
 *   buffers, transformed there and copied back, and the copies of one chunk
 *   overlap the kernel and the copies of its neighbours (two library streams,
 *   made by the first staged call on a device, plus `stream`). Pageable host
 *   memory works here (the copies then go through the driver's staging).
 * flags: QKNR_HOST_AUTO, QKNR_HOST_STAGED or QKNR_HOST_DIRECT.
 *
 * Asynchronous like qknr_apply: the work is ordered after everything
 * enqueued on `stream` before the call, and everything enqueued on `stream`
 * after it waits for the last result to reach the host. Synchronise `stream`
 * before reading h_q and h_k. Staged calls on one device are serialised on
 * the host (they share the library streams). Errors as qknr_apply, plus
 * QKNR_ERR_INVALID_ARG for a null host pointer, chunk_tokens < 0, an unknown
 * flag, or QKNR_HOST_DIRECT with a buffer the device cannot address.
 */
int qknr_apply_host(void *h_q, void *h_k, const void *q_w, const void *k_w,
                    const float *cos_sin_cache, const void *h_positions, void *d_q, void *d_k,
                    void *d_positions, int64_t num_tokens, int n_qo, int n_kv, int head_dim,
                    int rope_dim, int is_neox, int64_t q_stride, int64_t k_stride,
                    int64_t head_stride, float eps, int dtype, int64_t chunk_tokens, int flags,
                    void *stream);

/* kernels (QKNR_TUNE_KERNEL values and qknr_query_work_map out[0]) */
#define QKNR_KERNEL_AUTO 0     /* the measured rule (QKNR_TUNE_KERNEL only) */
#define QKNR_KERNEL_REGISTER 1 /* loads each warp item straight into registers */
#define QKNR_KERNEL_RING 2     /* double-buffers each warp's items in shared memory (cp.async) */

/* tuning keys for qknr_set_tuning / qknr_get_tuning (7 and 8 are not used) */
#define QKNR_TUNE_RESET 0       /* qknr_set_tuning(QKNR_TUNE_RESET, 0): every key back to automatic */
#define QKNR_TUNE_KERNEL 1      /* 0 auto (the rule: the ring kernel when items have 3 or 4 passes, the
                                   register kernel for decode-sized calls), 1 register, 2 ring */
#define QKNR_TUNE_PASSES 2      /* warp passes per item, 1..4 (0 auto: 4, or 1 when the whole call has
                                   at most 16 warp passes per SM) */
#define QKNR_TUNE_THREADS 3     /* threads per CTA, 64/128/256/512 (0 auto: 256; when no CTA cap is set,
                                   64 for the ring kernel's order 1 on interleaved calls and 512 for
                                   its order 2 when warps run at least 32 rounds of items) */
#define QKNR_TUNE_CTAS_PER_SM 4 /* cap on resident CTAs per SM (0 auto: occupancy) */
#define QKNR_TUNE_PDL 5         /* programmatic dependent launch: -1 auto (on), 0 off, 1 on */
#define QKNR_TUNE_RING_ORDER 6  /* ring kernel's issue order: 0 auto (2 for interleaved bf16 calls
                                   with head_dim 64, 128 or 256 whose warps run at least 6.5 rounds
                                   of items, else 1), 1 each item's successor issued as soon as the
                                   item's bytes land, 2 two items ahead after the first */
#define QKNR_TUNE_ORDER 9       /* item order: 0 auto (= 2), 1 a contiguous range per warp,
                                   2 interleaved (warp w takes items w, w + W, ...) */
#define QKNR_TUNE_PREFETCH 10   /* items per warp whose q/k rows (and the first positions) are
                                   prefetched into L2 while the kernel waits for the previous one
                                   on the stream: -1 none, 0 auto (4 for the register kernel, 1 for
                                   the ring kernel), 1..4 */

/*
 * Process-wide launch tuning, for benchmarks and tests; results do not depend
 * on it (every setting gives the same bits). Invalid values return
 * QKNR_ERR_INVALID_ARG and change nothing. The environment variable
 * QKNR_TUNE="kernel=2,ring_order=1,passes=4,threads=256,ctas=2,pdl=1,order=2,prefetch=1"
 * sets the same keys at first use.
 */
int qknr_set_tuning(int key, int value);
int qknr_get_tuning(int key, int *value);

/* Logging: with the environment variable QKNR_LOG=1, every distinct call shape
 * prints one line on stderr with the kernel, grid and work map chosen for it. */

/*
 * Measure the launch choices for one call shape and keep the fastest: for
 * later calls with exactly these sizes, strides and dtype (QKNR_INPUTS_READY
 * included) on the current device, qknr_apply, qknr_apply_checked and the
 * host and strided entry points use the chosen kernel, passes per item and
 * L2 prefetch depth instead of the fixed rule. Explicit qknr_set_tuning values
 * still take precedence. The op has no counterpart of this on the pages,
 * whose kernels fix their launch at compile time.
 *
 * The candidates (the register kernel and both orders of the ring kernel;
 * passes per item 4, 3, 2 or 1 where they chunk a token differently; prefetch
 * of 4, 2, 1 or no items) run on scratch buffers with the given layout, every
 * byte set to a constant nonzero value, never on the caller's data, each
 * timed with CUDA events over about 2 ms of launches in three alternating
 * rounds, beside the fixed rule's own launch. The one with the lowest median
 * time per launch is kept if it beats the rule's by more than 1% (the timing
 * noise); otherwise the rule's launch is kept. Input replicas rotate so that
 * no timed launch finds its inputs in L2.
 *
 * Arguments as for qknr_apply (num_tokens >= 1), without pointers. The call
 * allocates and frees its scratch (q and k at most 8 GiB, plus weights, a
 * cos|sin table of min(num_tokens, 65536) rows and positions), so it belongs
 * at set-up time, not on a hot path or inside a stream capture, and it waits
 * for `stream`. out (NULL allowed): QKNR_TUNE_FIELDS values, the chosen work
 * map as qknr_query_work_map reports it (out[0..12]), then out[13] the
 * measured time per launch in nanoseconds. A choice is kept until qknr_shutdown; tuning the
 * same shape again replaces it. Errors: QKNR_ERR_NOT_INITIALIZED,
 * QKNR_ERR_INVALID_ARG / UNSUPPORTED / MISALIGNED as qknr_apply would return
 * for the layout, QKNR_ERR_CUDA (scratch allocation or launch).
 */
int qknr_tune(int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim, int is_neox,
              int64_t q_stride, int64_t k_stride, int64_t head_stride, int dtype, void *stream,
              int64_t *out);

#define QKNR_WORK_MAP_FIELDS 13
#define QKNR_TUNE_FIELDS 14
/*
 * The launch qknr_apply would make for these sizes with contiguous q and k
 * (no launch, no pointers; assumes a 16-byte aligned cos|sin table), including
 * a choice qknr_tune made for that shape. out[QKNR_WORK_MAP_FIELDS]:
 *  0 kernel (QKNR_KERNEL_REGISTER or QKNR_KERNEL_RING)  1 grid CTAs
 *  2 threads per CTA  3 warp items  4 items per token  5 resident CTAs per
 *  SM  6 PDL on  7 warp passes per token  8 unroll class (most passes per
 *  item the instantiation holds: 2 or 4; the ring kernel's stage holds 4)
 *  9 item order (1 contiguous, 2 interleaved)  10 items per warp prefetched
 *    into L2 before the wait for the previous kernel  11 rope_dim compiled
 *    into the instantiation (0: read at run time; interleaved pairing with
 *    4-pass items has instantiations for rope_dim = head_dim and head_dim / 2
 *    at head_dim 64, 128 and 256)  12 ring kernel's issue order (1 or 2;
 *    0 for the register kernel)
 */
int qknr_query_work_map(int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim,
                        int is_neox, int dtype, int64_t *out);

#ifdef __cplusplus
}
#endif

#endif /* QKNR_H */

/*
 * detffn.h -- C ABI of libdetffn: a deterministic, bias-free gated BF16 FFN
 * (forward and backward) for NVIDIA GB300 (sm_103a).
 *
 * What it computes (RL-Kernel PR #325 "feat(ffn): add deterministic
 * distributed Triton FFN for ROCm", sections "Design" and "Operator test
 * matrix"):
 *
 *   gate = T(x, Wg), up = T(x, Wu)        contraction over K = H
 *   h    = bf16( bf16(SiLU(gate)) * up )   a BF16 stage boundary
 *   out  = T(h, Wd)                        contraction over K = I
 *
 * with Hugging Face [out, in] weights: Wg, Wu are [I, H]; Wd is [H, I].
 * T(A, B)[r, c] is the canonical FP32-leaf / BF16-node midpoint reduction
 * tree over K ("Design"): K is cut into contiguous leaves of leaf_width (64)
 * positions, each leaf is an FP32 partial sum, and leaves are combined by a
 * recursive midpoint split (left child = floor(n/2) leaves) in which every
 * internal node is rne_bf16(fp32(left) + fp32(right)).  The output element
 * is rne_bf16(root).  Because every contiguous K shard of a power-of-two
 * split is a subtree ("Make each contiguous TP K shard the same subtree used
 * by TP=1"), sharded and unsharded calls give the same bits.
 *
 * Conventions for every call below:
 *   - Tensors are row-major and contiguous, BF16 unless stated, in device
 *     memory owned by the caller.  The library allocates nothing per call;
 *     only detffn_create allocates (its tables and status word).
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Calls are asynchronous on that stream.  Argument
 *     errors are returned synchronously before anything is launched.
 *   - M == 0 (no tokens) or count == 0 returns DETFFN_OK and launches nothing.
 *   - Scratch memory is the caller's `ws` of `ws_bytes` bytes (256-byte
 *     aligned); query the size with detffn_workspace_size.
 *   - Results depend only on the inputs, the sizes and options->path; never
 *     on the shard count, the chunking, the stream or the run.
 */
#ifndef DETFFN_H
#define DETFFN_H

#include <stddef.h>

#if defined(__GNUC__)
#define DETFFN_API __attribute__((visibility("default")))
#else
#define DETFFN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DETFFN_OK = 0,
    DETFFN_ERR_INVALID_ARG = 1, /* NULL pointer, bad enum, overlapping buffers */
    DETFFN_ERR_SHAPE = 2,       /* sizes violate a precondition (e.g. shard rules) */
    DETFFN_ERR_ALIGN = 3,       /* a pointer is not aligned as the call requires */
    DETFFN_ERR_UNSUPPORTED = 4, /* option value not implemented (e.g. leaf_width != 64) */
    DETFFN_ERR_WORKSPACE = 5,   /* ws too small or not 256-byte aligned */
    DETFFN_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
    DETFFN_ERR_TIMEOUT = 7      /* a kernel's bounded wait ran out (read via detffn_get_status) */
} detffn_status;

typedef enum { DETFFN_F32 = 0, DETFFN_F16 = 1, DETFFN_BF16 = 2 } detffn_dtype;

/* Kernel family.  AUTO picks TENSOR when the tensor kernels cover the
 * call's contraction lengths (64-wide leaf counts of the form 1, 2^d or
 * 3*2^d, H and I multiples of 8, 16-byte-aligned tensors), else EXACT; it
 * never depends on the shard count or the chunking.  On the TENSOR family a
 * token's result does not depend on how many tokens the call has (1, a
 * decode batch, or a prefill of thousands: the same bits).
 * EXACT runs CUDA-core kernels whose leaves follow the LANE8x8 in-leaf
 * order (8 groups of 8 contiguous positions, each summed in ascending order
 * with fused multiply-adds from +0, then ((s0+s1)+(s2+s3))+((s4+s5)+(s6+s7)));
 * their results are bit-identical to a CPU evaluation of the same tree.
 * TENSOR computes each 64-wide leaf on the tensor cores (the hardware's own
 * in-leaf order) and applies the same tree to those leaves. */
typedef enum { DETFFN_PATH_AUTO = 0, DETFFN_PATH_EXACT = 1, DETFFN_PATH_TENSOR = 2 } detffn_path;

/* Option flags.  DETFFN_FLAG_TEST_STALL is for tests of the failure path
 * only: the call's streaming kernels issue no copies, so the first bounded
 * wait of every CTA runs out (after spin_limit polls: give a small one), the
 * CTAs stop with nothing in flight and the call's outputs are left
 * unfinished; detffn_get_status then returns DETFFN_ERR_TIMEOUT.  The fault
 * is made by withholding work, never by a bad address or a trap. */
enum {
    DETFFN_FLAG_TEST_STALL = 1,
    DETFFN_FLAG_OVERLAP_DHIDDEN = 2,
    DETFFN_FLAG_SPLIT_FORWARD = 4,
    DETFFN_FLAG_HOST_IO = 8
};
/* DETFFN_FLAG_OVERLAP_DHIDDEN (detffn_backward with options->shards = k > 1;
 * PR #325, "Communication overlap assessment"): the rank tree of the gate
 * contribution's shard roots runs on a second stream of the handle while the
 * up contribution's shards are computed on `stream`; the gate-then-up
 * addition waits for both.  The bits are those of the one-stream call.
 * Without shards it changes nothing.
 * DETFFN_FLAG_SPLIT_FORWARD (detffn_forward): on the tensor family with at
 * most 32 tokens the forward is one launch (PR #325, "Communication overlap
 * assessment": the gate/up to down dependency taken per K range of the down
 * projection, inside the launch) wherever the shape allows; this flag asks
 * for the two-launch form instead (gate/up with SiLU * up, then down).  The
 * bits are the same.
 * DETFFN_FLAG_HOST_IO (detffn_forward, detffn_forward_sharded, and
 * detffn_workspace_size for their ops): x and out are page-locked host
 * buffers of this process (cudaHostAlloc, or registered with
 * cudaHostRegister); the weights, gate_save, up_save and ws stay device
 * memory.  The call reads x over the host link into the workspace and writes
 * out back to the host buffer with its own copy kernels, on `stream` and in
 * stream order (no host synchronization inside the call: out is complete
 * once the stream has reached the end of the call).  The workspace must be
 * sized with the flag (it holds the two staged copies).  x or out not
 * page-locked host memory: DETFFN_ERR_INVALID_ARG.  The bits are those of
 * the call on device buffers.  Other calls: DETFFN_ERR_INVALID_ARG. */

typedef struct {
    int leaf_width;        /* 64; anything else returns DETFFN_ERR_UNSUPPORTED */
    int path;              /* detffn_path */
    int shards;            /* detffn_backward only: k in {1,2,4,8} TP shards of I for dHidden */
    int flags;             /* DETFFN_FLAG_* bits (0: none); other bits: DETFFN_ERR_INVALID_ARG */
    long long spin_limit;  /* polls before a role's bounded in-kernel wait gives up; 0 = default
                              (2^26).  Waits that drain a CTA's own copies and tensor-core work
                              before it exits always use the default. */
} detffn_options;          /* pass NULL for {64, AUTO, 1, 0, 0} */

typedef struct detffn_handle_s *detffn_handle;

/* Operation codes for detffn_workspace_size. */
enum {
    DETFFN_OP_FORWARD = 0,
    DETFFN_OP_FORWARD_SHARDED = 1,
    DETFFN_OP_BACKWARD = 2,
    DETFFN_OP_WGRAD_CHUNKED = 3
};

/* Creates a handle bound to CUDA device `device`: builds the SiLU tables
 * (correctly rounded BF16 SiLU and FP32 SiLU' for all 2^16 gate values), a
 * device status word and the tree tickets of the few-token kernels (4 KiB:
 * where a tree's K range is split over several CTAs, the last of them to
 * finish folds their subtree roots into the root).  *out is set only on
 * success.  The handle may be used from one host thread at a time, and its
 * calls must run in order on the GPU (one stream, or streams ordered by
 * events): calls through one handle that overlap on the GPU share the status
 * word and the tickets and must not be issued. */
DETFFN_API detffn_status detffn_create(detffn_handle *out, int device);

/* Frees the handle's device memory; waits for nothing.  NULL is accepted. */
DETFFN_API detffn_status detffn_destroy(detffn_handle h);

/* Scratch bytes a call needs for (op, M, H, I, k); k is the shard count for
 * DETFFN_OP_FORWARD_SHARDED and DETFFN_OP_BACKWARD (1 otherwise), and M is
 * the total token count for DETFFN_OP_WGRAD_CHUNKED. */
DETFFN_API detffn_status detffn_workspace_size(detffn_handle h, int op, long long M, long long H,
                                    long long I, int k, const detffn_options *opts,
                                    size_t *bytes);

/* Forward (PR #325, "Design"; "Operator test matrix").
 *   x [M,H], Wg [I,H], Wu [I,H], Wd [H,I] (inputs); out [M,H] (output).
 *   gate_save, up_save: NULL for inference, or [M,I]
 *   buffers that receive gate and up (training mode).  out is bit-identical
 *   either way ("Repeated execution and training/inference forward: 0 mismatch",
 *   "Correctness results").  Outputs must not overlap inputs. */
DETFFN_API detffn_status detffn_forward(detffn_handle h, const void *x, const void *Wg, const void *Wu,
                             const void *Wd, void *out, void *gate_save, void *up_save,
                             long long M, long long H, long long I,
                             void *ws, size_t ws_bytes, void *stream,
                             const detffn_options *opts);

/* Forward with tensor-parallel emulation on one GPU (PR #325, "Design": "Make
 * each contiguous TP K shard the same subtree used by TP=1" and "fixed
 * balanced BF16 rank reduction tree").  Shard s in [0,k) owns rows
 * [s*I/k, (s+1)*I/k) of Wg and Wu and the same columns of Wd; it computes its
 * gate/up/h slice and the subtree root p_s [M,H] of the down projection over
 * its I/k positions into ws; then out = ((p0+p1)+(p2+p3))+... with BF16
 * nodes.  k in {1,2,4,8}; requires I % k == 0, (I/k) % 64 == 0 and
 * (I/k)/64 >= 2 for k > 1 (a one-leaf shard root would be an unrounded FP32
 * leaf), else DETFFN_ERR_SHAPE.  out equals detffn_forward's out bit for bit. */
DETFFN_API detffn_status detffn_forward_sharded(detffn_handle h, const void *x, const void *Wg,
                                     const void *Wu, const void *Wd, void *out,
                                     void *gate_save, void *up_save,
                                     long long M, long long H, long long I, int k,
                                     void *ws, size_t ws_bytes, void *stream,
                                     const detffn_options *opts);

/* Backward (PR #325, "Design"; "Communication overlap assessment" for the
 * gate-then-up order).  Inputs: x [M,H], the weights, gate and up [M,I]
 * saved by a training forward, dOut [M,H].  Outputs (overwritten, never
 * accumulated): dX [M,H], dWg [I,H], dWu [I,H], dWd [H,I].
 *   dh = T(dOut, Wd^T) over K=H
 *   dU = bf16(dh*a), dA = bf16(dh*u), dG = bf16(fp32(dA*SiLU'(g)))   a = bf16(SiLU(g))
 *   cg = T(dG, Wg^T), cu = T(dU, Wu^T) over K=I; dX = bf16(cg + cu)
 *   dWd = T(dOut^T, h^T), dWg = T(dG^T, x^T), dWu = T(dU^T, x^T) over K=M,
 *   with h = bf16(a*u) recomputed.
 * opts->shards = k > 1 computes cg and cu as k shard subtree roots combined by
 * the rank tree (same bits).  dh_save, dU_save, dG_save: optional [M,I]
 * buffers that receive those stages (NULL to skip). */
DETFFN_API detffn_status detffn_backward(detffn_handle h, const void *x, const void *Wg, const void *Wu,
                              const void *Wd, const void *gate, const void *up,
                              const void *dOut, void *dX, void *dWg, void *dWu, void *dWd,
                              void *dh_save, void *dU_save, void *dG_save,
                              long long M, long long H, long long I,
                              void *ws, size_t ws_bytes, void *stream,
                              const detffn_options *opts);

/* Weight gradients from a token set given as n_chunks chunks in logical token
 * order (context-parallel emulation; PR #325, "Design": "Gather complete CP
 * token sequences before weight-gradient GEMMs so their K tree matches
 * CP=1").  Host arrays of length n_chunks: chunk_tokens[c] >= 0 and device
 * pointers x_chunks[c] [t_c,H], gate_chunks[c] [t_c,I], up_chunks[c] [t_c,I],
 * dOut_chunks[c] [t_c,H].  The row-wise stages (dh, dU, dG, h) run per chunk
 * with the path chosen from the total token count; the chunks are gathered
 * into ws in order and the weight gradients are one tree over all tokens, so
 * dWg [I,H], dWu [I,H], dWd [H,I] equal detffn_backward's bit for bit for any
 * chunking. */
DETFFN_API detffn_status detffn_wgrad_chunked(detffn_handle h, int n_chunks, const long long *chunk_tokens,
                                   const void *const *x_chunks, const void *const *gate_chunks,
                                   const void *const *up_chunks, const void *const *dOut_chunks,
                                   const void *Wd, void *dWg, void *dWu, void *dWd,
                                   long long H, long long I, void *ws, size_t ws_bytes,
                                   void *stream, const detffn_options *opts);

/* Rank-tree reduction (PR #357 "optimize deterministic ROCm collectives with
 * HIP IPC", "Design"; PR #356 "add deterministic ROCm/RCCL transport
 * collectives", "Design"): out[e] = ((b0+b1)+(b2+b3))+((b4+b5)+(b6+b7)) for
 * n in {1,2,4,8} device buffers of `count` elements of `dtype`; every node
 * is an FP32 add rounded (to nearest even) to dtype.  `inputs` is a HOST
 * array of n device pointers.  Any element alignment is accepted (offset
 * views); 16-byte-aligned buffers take a vector path, 4-byte-aligned 16-bit
 * buffers a two-element path, the rest a scalar path.  out may be exactly
 * one of the inputs (in place); any other overlap is DETFFN_ERR_INVALID_ARG.
 * count == 0 launches nothing. */
DETFFN_API detffn_status detffn_rank_tree_reduce(const void *const *inputs, int n, void *out,
                                      long long count, int dtype, void *stream);

/* One tree contraction, the building block of every call above:
 * out[r*o_rs + c] = T_K(A[r*a_rs + k*a_ks], B[c*b_rs + k*b_ks]) in BF16, for
 * r < R, c < C (element strides, any layout).  K == 0 writes +0. */
DETFFN_API detffn_status detffn_tree_gemm(detffn_handle h, const void *A, long long a_rs, long long a_ks,
                               const void *B, long long b_rs, long long b_ks,
                               long long R, long long C, long long K,
                               void *out, long long o_rs, void *stream,
                               const detffn_options *opts);

/* Leaf dump (a diagnostic of the TENSOR family: it lets a test apply the
 * canonical tree to the tensor cores' own leaves; RL-Kernel PR #325,
 * "Design"): the same contraction as
 * detffn_tree_gemm on the tensor family (same kernels, same plan, same
 * bits in `out`), which also writes every FP32 leaf to `leaves`, a device
 * array of R * C * L floats laid out [R][C][L], L = ceil(K / 64).  Applying
 * the canonical tree to these leaves gives `out` exactly; each leaf is the
 * tensor core's sum of its 64 (or fewer) products.  K >= 1; EXACT returns
 * DETFFN_ERR_UNSUPPORTED (its leaves follow the documented LANE8x8 order),
 * shapes the tensor family does not cover return DETFFN_ERR_UNSUPPORTED.
 * The dump is slow (scattered 4-byte stores) and meant for tests. */
DETFFN_API detffn_status detffn_tree_gemm_leaves(detffn_handle h, const void *A, long long a_rs,
                                      long long a_ks, const void *B, long long b_rs, long long b_ks,
                                      long long R, long long C, long long K, void *out, long long o_rs,
                                      void *leaves, void *stream, const detffn_options *opts);

/* Copies the handle's SiLU tables to host memory: silu_bf16[65536] (BF16 bit
 * patterns) and dsilu_f32[65536], indexed by the gate's bit pattern.  Either
 * pointer may be NULL. */
DETFFN_API detffn_status detffn_silu_tables(detffn_handle h, unsigned short *silu_bf16, float *dsilu_f32);

/* Per-kernel timing for measurement.  detffn_profiling(h, 1) clears the
 * records and makes every later launch through h record a CUDA event pair on
 * the launch's own stream, with the kernel's name and its algorithmic bytes
 * and flops (operands read once, outputs written once); detffn_profiling(h, 0)
 * stops recording.  detffn_profile_read synchronises the device, sums the
 * records per kernel name into out[0..*n) (at most `max` entries), and clears
 * them.  Profiling adds an event record between launches and nothing else. */
typedef struct {
    char name[48];
    int launches;
    double ms;     /* summed event-measured durations */
    double bytes;  /* summed algorithmic bytes */
    double flops;  /* summed algorithmic flops */
} detffn_kernel_time;

DETFFN_API detffn_status detffn_profiling(detffn_handle h, int enable);
DETFFN_API detffn_status detffn_profile_read(detffn_handle h, int max, detffn_kernel_time *out, int *n);

/* Decode forward that allocates nothing (the pages have no counterpart to
 * this call; it exists for callers that cannot call cudaMalloc, such as a
 * process whose device memory is already owned by a caching allocator's
 * pool, or a runtime that only hands out buffers reserved in advance).
 * It computes exactly what detffn_forward computes on the EXACT path -- the
 * same bits -- for 1 <= M <= 8 tokens and H, I in {256, 512, 1024, 2048,
 * 4096} or {768, 1536, 3072, 6144, 12288} (4 to 64 leaves of 64, a power of
 * two, or 12 to 192, three times one).  Inputs x [M,H] and the weights must
 * be 16-byte aligned; out [M,H] is written.  Other sizes return
 * DETFFN_ERR_SHAPE, misaligned pointers DETFFN_ERR_ALIGN, and nothing is
 * launched.
 * Its scratch (h, the kernels' block-root planes and tickets, and a status
 * word; about 3.3 MiB) and its SiLU table are fixed-size arrays inside the
 * library, held by every GPU that loads it until the process exits.  The
 * first call on a device performs a one-time set-up there (it resolves those
 * arrays' device addresses and copies the SiLU table with a synchronous
 * cudaMemcpy); make that first call before any stream capture.  Every call
 * uses the same arrays and first clears what must start at zero (the tickets
 * and the status word), so calls that overlap on the GPU (on different
 * streams, or from different host threads) race and must not be issued;
 * calls in order on one stream are fine.  It uses the current device and runs
 * on `stream` (a cudaStream_t).  A bounded in-kernel wait that runs out is
 * reported by detffn_forward_decode_noalloc_status, not by this call. */
DETFFN_API detffn_status detffn_forward_decode_noalloc(const void *x, const void *Wg,
                                                       const void *Wu, const void *Wd, void *out,
                                                       long long M, long long H, long long I,
                                                       void *stream);

/* Status of the allocation-free decode forward on the current device:
 * synchronises `stream`, then returns and clears the status word of the
 * last detffn_forward_decode_noalloc call (DETFFN_OK, or DETFFN_ERR_TIMEOUT
 * when a bounded wait ran out: its out is then unfinished).  Allocates
 * nothing; may perform the same one-time set-up as the first call. */
DETFFN_API detffn_status detffn_forward_decode_noalloc_status(void *stream);

/* For tests of the failure path only: later detffn_forward_decode_noalloc
 * calls in this process poll their bounded waits at most spin_limit times
 * (0: the default bound) and, with stall = 1, issue no copies, so that their
 * first wait runs out and the status word reports DETFFN_ERR_TIMEOUT without
 * any fault.  (0, 0), the state at load, is the normal path.  A negative
 * spin_limit or another stall value: DETFFN_ERR_INVALID_ARG. */
DETFFN_API detffn_status detffn_forward_decode_noalloc_test_waits(long long spin_limit, int stall);

/* Diagnostic: out[i] = the BF16 rounding (to nearest, ties to even) of the
 * FP32 value in[i], computed on the device with the very conversion every
 * kernel of the library uses for leaves, nodes and stage boundaries; a test
 * compares it with an independent rounding rule over all 2^32 patterns.
 * in: n floats, out: n BF16 (device, 4- and 2-byte aligned, not overlapping). */
DETFFN_API detffn_status detffn_cvt_f32_bf16(detffn_handle h, const void *in, void *out, long long n,
                                             void *stream);

/* Diagnostic: counts the BF16 pairs (a, b), over all 2^32 of them, for which
 * the device's packed add.rn.bf16x2 differs from the tree node
 * rne_bf16(fp32(a) + fp32(b)) (any NaN equals any NaN).  The tree's higher
 * nodes use the packed add only if this is 0 (the two are the same rounding
 * of a + b, since binary32 has more than 2*8+2 significand bits).  Allocates
 * an 8-byte counter and synchronises the device. */
DETFFN_API detffn_status detffn_selfcheck_node_add(detffn_handle h, unsigned long long *mismatches);

/* Diagnostic, host only (no device, no handle): checks the decomposition of
 * K ranges into pieces used by the few-token tensor kernels (balanced K
 * ranges; RL-Kernel PR #325, "Design": every contiguous range of leaves that
 * is an aligned block is a subtree of the canonical tree).  For every tile of
 * 2^E bottom groups, E <= max_levels (at most 8): the closed-form pieces of
 * every group range equal the greedy decomposition into maximal aligned
 * blocks, and for every split of the tile into three consecutive ranges the
 * pieces, folded left to right with their fold codes, pair each right child
 * with its left sibling and end in the tile's root exactly once.  Writes the
 * number of failed cases to *failures.  DETFFN_ERR_INVALID_ARG for a null
 * pointer or max_levels outside [0, 8]. */
DETFFN_API detffn_status detffn_selfcheck_pieces(int max_levels, unsigned long long *failures);

/* Host check (no GPU needed) of the one-launch decode forward's schedule
 * (see DETFFN_FLAG_SPLIT_FORWARD) over a grid of shapes (H, I in
 * {256, ..., 12288}) and SM counts: each down-projection block runs on
 * exactly one CTA, each range of I counts exactly the gate/up tiles whose
 * columns of h its blocks read, the waiter counts match, the blocks tile each
 * tree's K axis, and the fold fits the pipeline stages.  Writes the shapes
 * covered to *cases and the failed ones to *failures; DETFFN_ERR_INVALID_ARG
 * for a null pointer. */
DETFFN_API detffn_status detffn_selfcheck_fused_schedule(unsigned long long *cases,
                                                         unsigned long long *failures);

/* Synchronises `stream`, then returns and clears the handle's device status
 * word (DETFFN_OK or DETFFN_ERR_TIMEOUT from a bounded wait).  The word is
 * sticky: once a wait has run out, every later streaming kernel launched
 * through the handle returns at entry (leaving its outputs unwritten) until
 * this call clears it, so no kernel builds on another's unfinished output.
 * On DETFFN_ERR_TIMEOUT it also clears the tree tickets (a stopped launch
 * may have left some taken), so that the next call starts clean. */
DETFFN_API detffn_status detffn_get_status(detffn_handle h, void *stream);

/* The CUDA error behind the calling thread's last DETFFN_ERR_CUDA (a static
 * string); reading it clears it. */
DETFFN_API const char *detffn_last_cuda_error(void);

/* Static description of a status code. */
DETFFN_API const char *detffn_status_string(detffn_status s);

#ifdef __cplusplus
}
#endif

#endif /* DETFFN_H */

/*
 * tp.h -- C ABI of the B300 (sm_103a) tensor-parallel sharded linear library.
 *
 * What it computes.  For a linear map Y = X W with X [M, K], W [K, Nout]
 * (chipfoundryservices.com topic page "Tensor Parallelism", section "Tensor
 * Parallelism Fundamentals"), the weight is split into n_shards logical
 * shards that all live in the memory of ONE GPU:
 *
 *   - split by output columns, W = [W_0, ..., W_{n-1}]: shard i computes
 *     Y_i = X W_i and the shard outputs are concatenated (same page, section
 *     "Column-Wise Parallelism"; aiforbusinessandlife.com glossary
 *     "Tensor Parallelism", section "Worked example");
 *   - split by the contracted rows, W = [W_0; ...; W_{n-1}] with X split to
 *     match: shard i computes the partial X_i W_i and the partials are added
 *     (topic page, section "Row-Wise Parallelism"; glossary "Worked example");
 *   - the MLP block chains the two with an activation applied per shard and
 *     no exchange in between (topic page, section "Megatron-LM Tensor
 *     Parallelism", MLP layer splitting).
 *
 * The exchanges of a multi-device system become on-device operations: the
 * all-gather is a concat (fused into the GEMM's output store, or the
 * standalone tp_shard_concat) and the all-reduce is a sum (fused into the
 * GEMM's fp32 accumulator, or the standalone tp_shard_reduce).
 *
 * Conventions shared by every entry point:
 *   - Matrices are dense and row-major with no padding: element (r, c) of an
 *     [R, C] matrix is at offset r*C + c.
 *   - Every data pointer is a DEVICE pointer on the current CUDA device.  The
 *     caller owns all memory, including the MLP workspace; the library never
 *     allocates device memory and keeps no per-call state.
 *   - Every call is asynchronous on stream `s` (0 = legacy default stream).
 *     Arguments are validated on the host before any launch; a validation
 *     error returns synchronously and launches nothing.  A failed launch
 *     returns TP_ERR_CUDA.
 *   - bf16 inputs take the tensor-core path (tcgen05 + TMA), which needs
 *     16-byte aligned base pointers and row pitches that are multiples of 16
 *     bytes (K and Nout multiples of 8).  fp32 inputs take a CUDA-core path
 *     with exact fp32 fused multiply-adds in ascending k (bit-exact for
 *     integer-valued data whose sums stay below 2^24); it needs only 4-byte
 *     alignment.  M may be anything >= 0.
 *   - Each of M, K, Nout (d, f) is at most 2^31 - 1 and each matrix holds at
 *     most 2^40 elements; larger sizes return TP_ERR_SHAPE (the workspace
 *     size queries return 0 for them).
 *   - Outputs must not overlap inputs (TP_ERR_ALIAS).
 *   - Device-side waits are bounded; a wait that runs out marks the device
 *     status word, read back with tp_get_device_status().
 */
#ifndef TP_B300_H
#define TP_B300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>   /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TP_OK = 0,
    TP_ERR_NULL = 1,          /* a required pointer is NULL */
    TP_ERR_SHAPE = 2,         /* negative size, sizes inconsistent, a size
                                 above 2^31 - 1, or a matrix of more than
                                 2^40 elements */
    TP_ERR_DIVISIBILITY = 3,  /* the split axis is not divisible by n_shards
                                 (or by col_groups), or n_shards out of range */
    TP_ERR_ALIGNMENT = 4,     /* pointer or row pitch not aligned as required */
    TP_ERR_DTYPE = 5,         /* unsupported dtype combination */
    TP_ERR_WORKSPACE = 6,     /* workspace NULL or smaller than required */
    TP_ERR_CUDA = 7,          /* a CUDA runtime/driver call failed */
    TP_ERR_DEVICE_TIMEOUT = 8,/* a bounded device-side wait ran out */
    TP_ERR_ALIAS = 9          /* an output overlaps an input */
} tp_status;

typedef enum { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;
typedef enum { TP_SPLIT_COLS = 0, TP_SPLIT_ROWS = 1 } tp_split;   /* split axis of W */
typedef enum { TP_ACT_NONE = 0, TP_ACT_GELU = 1 } tp_act;

/* Largest shard count accepted by any entry point. */
#define TP_MAX_SHARDS 64

/*
 * Column-parallel linear (topic page, "Column-Wise Parallelism").
 *
 *   Y[M, Nout] = act(X[M, K] . W[K, Nout]),  W = [W_0 | ... | W_{n-1}],
 *   W_i = columns [i*Nout/n, (i+1)*Nout/n).
 *
 * Shard i computes Y_i = act(X W_i) with act applied to each shard on its own
 * (act = TP_ACT_GELU: exact GeLU x*Phi(x), evaluated in fp32 with an
 * error below 1e-4 of the value over the whole range, the negative tail
 * included; a bf16 output is within one ulp of the correctly rounded GeLU).
 *   Y         optional: the concatenated output [M, Nout] -- the concat is
 *             fused into the output store, so no extra pass is made.
 *   Y_shards  optional: the shard outputs kept apart, [n_shards, M, Nout/n].
 * At least one of Y, Y_shards must be non-NULL; both may be given.
 *   in_t      dtype of X and W (TP_BF16: tensor cores, fp32 accumulation;
 *             TP_F32: CUDA cores, fp32 accumulation).
 *   out_t     dtype of Y and Y_shards (bf16 results are rounded to nearest
 *             even from the fp32 accumulator).
 * The result of every output element does not depend on n_shards: the
 * concatenated Y is bit-identical to the n_shards = 1 call.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_DIVISIBILITY (Nout % n_shards),
 * TP_ERR_ALIGNMENT, TP_ERR_DTYPE, TP_ERR_ALIAS, TP_ERR_CUDA.
 */
tp_status tp_column_linear(const void *X, const void *W, void *Y, void *Y_shards,
                           int64_t M, int64_t K, int64_t Nout, int n_shards,
                           tp_dtype in_t, tp_dtype out_t, tp_act act, cudaStream_t s);

/*
 * Column-parallel linear with a head-group split (topic page, SVG figure
 * panel "Attention Head Parallelism": each device owns a subset of heads;
 * section "Megatron-LM Tensor Parallelism": Q, K, V projections are split by
 * columns).  The Nout columns form col_groups equal blocks (Q | K | V for a
 * fused QKV weight); shard i owns slice i of every block:
 *   gw = Nout/col_groups, sw = gw/n_shards,
 *   shard i owns columns { b*gw + i*sw + j : b < col_groups, j < sw },
 * and its local output Y_shards[i] is [M, col_groups*sw] ordered block by
 * block.  Y (if given) is the full output in W's own column order.
 * col_groups = 1 is tp_column_linear.  Extra error: TP_ERR_DIVISIBILITY if
 * Nout % col_groups or gw % n_shards is non-zero.
 */
tp_status tp_column_linear_grouped(const void *X, const void *W, void *Y, void *Y_shards,
                                   int64_t M, int64_t K, int64_t Nout, int n_shards,
                                   int col_groups, tp_dtype in_t, tp_dtype out_t,
                                   tp_act act, cudaStream_t s);

/*
 * Row-parallel linear (topic page, "Row-Wise Parallelism"; glossary "How it
 * works": splitting the contracted dimension gives partials to be summed).
 *
 *   Y[M, Nout] = sum_{i=0}^{n-1} X[:, K_i] . W[K_i, :],
 *   K_i = [i*K/n, (i+1)*K/n),
 *
 * summed in ascending shard order in fp32.
 *   P_out == NULL: the partials are never materialised -- every shard's
 *     product is accumulated into the same fp32 tensor-memory accumulator
 *     (or, when the output has too few tiles to fill the GPU, the first and
 *     the second half of the shards are accumulated by the two CTA pairs of
 *     one thread-block cluster and the two fp32 sums are added once,
 *     exchanged between the pairs' shared memories).  Y is required.
 *   P_out != NULL: the fp32 partials are written to P_out [n_shards, M, Nout];
 *     if Y is also non-NULL it is then formed from them by tp_shard_reduce.
 * Errors: as tp_column_linear, with TP_ERR_DIVISIBILITY for K % n_shards.
 * The bf16 path with P_out needs K/n_shards to be a multiple of 8.
 */
tp_status tp_row_linear(const void *X, const void *W, void *Y, float *P_out,
                        int64_t M, int64_t K, int64_t Nout, int n_shards,
                        tp_dtype in_t, tp_dtype out_t, cudaStream_t s);

/*
 * Biased variants.  The pages write Y = X W throughout and mention biases
 * only among the parameters a device holds a part of (Manning liveBook
 * concept page "Tensor parallelism": each device works on part of a linear
 * layer's weights and biases); the reading taken: a column-split bias b [Nout] is split
 * with W's columns and each shard adds its slice to its own outputs (before
 * the activation); a row-split bias is added ONCE, after the shards'
 * partials are summed -- added by every shard it would be counted n_shards
 * times.
 *   bias: device pointer to Nout values of in_t, or NULL (then these are
 *   exactly tp_column_linear / tp_row_linear); 16-byte aligned for bf16.
 *   tp_row_linear_bias with P_out: the partials stay bias-free and the bias
 *   is added by the reduce that forms Y.
 * Errors: as the unbiased calls; TP_ERR_ALIAS if an output overlaps bias.
 */
tp_status tp_column_linear_bias(const void *X, const void *W, const void *bias, void *Y,
                                void *Y_shards, int64_t M, int64_t K, int64_t Nout, int n_shards,
                                tp_dtype in_t, tp_dtype out_t, tp_act act, cudaStream_t s);
tp_status tp_row_linear_bias(const void *X, const void *W, const void *bias, void *Y,
                             float *P_out, int64_t M, int64_t K, int64_t Nout, int n_shards,
                             tp_dtype in_t, tp_dtype out_t, cudaStream_t s);

/*
 * Either split, chosen by `split` (glossary "Check your understanding":
 * different output coordinates are concatenated, the same coordinates are
 * added).  TP_SPLIT_COLS calls tp_column_linear(X, W, Y, NULL, ...);
 * TP_SPLIT_ROWS calls tp_row_linear(X, W, Y, NULL, ...) and requires
 * act == TP_ACT_NONE (an activation of a partial sum is not the activation of
 * the sum; TP_ERR_DTYPE otherwise).
 */
tp_status tp_sharded_linear(const void *X, const void *W, void *Y,
                            int64_t M, int64_t K, int64_t Nout, int n_shards,
                            tp_split split, tp_dtype in_t, tp_dtype out_t,
                            tp_act act, cudaStream_t s);

/*
 * Standalone all-reduce as an on-device sum (topic page, "Row-Wise
 * Parallelism", output combination).
 *   P  fp32 partials [n_shards, rows, cols].
 *   Y  [rows, cols] of out_t:  Y[r, c] = sum_{i=0}^{n-1} P[i, r, c], added in
 *      fp32 in ascending i, then rounded to nearest even if out_t = TP_BF16.
 *      NaN and Inf propagate.
 * P and Y need 16-byte alignment.  Errors: TP_ERR_NULL, TP_ERR_SHAPE,
 * TP_ERR_DIVISIBILITY (n_shards out of [1, TP_MAX_SHARDS]), TP_ERR_ALIGNMENT,
 * TP_ERR_DTYPE, TP_ERR_ALIAS, TP_ERR_CUDA.
 */
tp_status tp_shard_reduce(const float *P, void *Y, int64_t rows, int64_t cols, int n_shards,
                          tp_dtype out_t, cudaStream_t s);

/*
 * Standalone all-gather as an on-device concat (topic page, "Column-Wise
 * Parallelism", output combination).
 *   Ys  shard outputs [n_shards, rows, shard_cols] of dtype t.
 *   Y   [rows, n_shards*shard_cols]: Y[:, i*shard_cols + j] = Ys[i, :, j].
 * The copy moves 16-byte vectors, so shard_cols must be a multiple of 8
 * (bf16) or 4 (fp32) and both pointers 16-byte aligned.
 */
tp_status tp_shard_concat(const void *Ys, void *Y, int64_t rows, int64_t shard_cols,
                          int n_shards, tp_dtype t, cudaStream_t s);

/*
 * QKV projection with grouped-query attention heads (topic page, SVG figure,
 * "Attention Head Parallelism": split the Q heads evenly, replicate the
 * shared KV heads).
 *
 *   W = [Wq | Wk | Wv] [K, (n_q_heads + 2 n_kv_heads) * head_dim], head h of
 *   each block in columns [h*head_dim, (h+1)*head_dim) of that block.
 *   Shard i owns Q heads [i*n_q/n, (i+1)*n_q/n) and the KV heads its Q heads
 *   read: [i*n_kv/n, (i+1)*n_kv/n) when n divides n_kv (split), the single
 *   head floor(i*n_kv/n) when n_kv divides n (held by n/n_kv shards).
 *   Y [M, (n_q + 2 n_kv) * head_dim]: the full projection X W (required;
 *     the KV heads are computed once, not once per holder).
 *   Y_shards (optional) [n, M, (n_q/n + 2 kvs) * head_dim], kvs = KV heads
 *     per shard: shard i's local [Q_i | K_i | V_i], copied from Y with TMA
 *     boxes (a replicated KV head lands in every shard that holds it);
 *     head_dim * sizeof(out_t) must be a multiple of 16.
 * With n_kv_heads == n_q_heads this is tp_column_linear_grouped with
 * col_groups = 3.  Errors: TP_ERR_SHAPE if n_kv_heads does not divide
 * n_q_heads or 3*n_shards > 192; TP_ERR_DIVISIBILITY if n does not divide
 * n_q_heads or neither of n, n_kv_heads divides the other; as
 * tp_column_linear otherwise.
 */
tp_status tp_qkv_linear(const void *X, const void *W, void *Y, void *Y_shards, int64_t M,
                        int64_t K, int64_t n_q_heads, int64_t n_kv_heads, int64_t head_dim,
                        int n_shards, tp_dtype in_t, tp_dtype out_t, cudaStream_t s);

/*
 * Concat for the head-group split: shard i's local columns are col_groups
 * blocks of sw = shard_cols/col_groups columns; block b lands at output
 * columns [b*gw + i*sw, b*gw + (i+1)*sw) with gw = n_shards*sw (the inverse
 * of tp_column_linear_grouped's ownership).  sw must be a multiple of 8
 * (bf16) or 4 (fp32).
 */
tp_status tp_shard_concat_grouped(const void *Ys, void *Y, int64_t rows, int64_t shard_cols,
                                  int n_shards, int col_groups, tp_dtype t, cudaStream_t s);

/*
 * Bytes of workspace tp_mlp_block needs for M tokens and intermediate width
 * f with inputs of dtype t: the hidden activation H [M, f] in dtype t,
 * rounded up to 256 bytes.  Returns 0 for negative sizes.
 */
size_t tp_mlp_block_workspace_size(int64_t M, int64_t f, tp_dtype t);

/*
 * Megatron-style MLP block (topic page, "Megatron-LM Tensor Parallelism",
 * MLP layer splitting; "Row-Wise Parallelism": the second layer's input is
 * already split by the first):
 *
 *   H_i = GeLU(X . W1_i)           W1_i = columns [i*f/n, (i+1)*f/n) of W1
 *   Y   = sum_i H_i . W2_i         W2_i = rows    [i*f/n, (i+1)*f/n) of W2
 *
 *   X [M, d], W1 [d, f], W2 [f, d], Y [M, d] (out_t).
 *   ws, ws_bytes: caller-owned device workspace of at least
 *     tp_mlp_block_workspace_size(M, f, in_t) bytes, 16-byte aligned.  H is
 *     stored there in in_t (bf16 H is rounded to nearest even from the fp32
 *     GeLU output); it stays partitioned by shard -- H_i is the column block
 *     i of H -- and is never gathered.
 * Two kernels on stream s: the column GEMM with the GeLU fused into its
 * epilogue, then the row GEMM with the shard sum fused into its fp32
 * accumulator (the second launched so that its set-up overlaps the first's
 * tail).
 * Errors: as the two linears, plus TP_ERR_WORKSPACE.
 */
tp_status tp_mlp_block(const void *X, const void *W1, const void *W2, void *Y,
                       void *ws, size_t ws_bytes,
                       int64_t M, int64_t d, int64_t f, int n_shards,
                       tp_dtype in_t, tp_dtype out_t, cudaStream_t s);

/*
 * MLP block with biases: Y = sum_i GeLU(X W1_i + b1_i) W2_i + b2, b1 [f]
 * split with W1's columns (each shard adds its slice before the GeLU), b2
 * [d] added once after the sum.  b1 or b2 may be NULL.  Otherwise as
 * tp_mlp_block.
 */
tp_status tp_mlp_block_bias(const void *X, const void *W1, const void *b1, const void *W2,
                            const void *b2, void *Y, void *ws, size_t ws_bytes, int64_t M,
                            int64_t d, int64_t f, int n_shards, tp_dtype in_t, tp_dtype out_t,
                            cudaStream_t s);

/*
 * MLP block without a caller-provided workspace.  (No counterpart on the
 * pages: this is a property of the library's memory handling, not of the
 * method.)
 *
 * Same computation, arguments and errors as tp_mlp_block, minus ws and
 * ws_bytes.  It is meant for callers that cannot allocate device memory when
 * they call: a serving loop that must not call cudaMalloc once it is running
 * (cudaMalloc can synchronise the whole device and stall other streams), or
 * a host framework that owns all device memory through its own pool and
 * hands the library only its input and output tensors.  The hidden
 * activation H is kept instead in a fixed array inside the library's device
 * image, TP_STATIC_WS_BYTES bytes, which every GPU that loads the library
 * holds until the process exits.  The call allocates nothing.
 *   - Limit: M * f * sizeof(in_t) <= TP_STATIC_WS_BYTES (32 MiB: for bf16,
 *     for example, M = 2048 tokens with f up to 8192); larger problems
 *     return TP_ERR_WORKSPACE without launching anything.
 *   - The first call on a device looks up the array's device address on
 *     that device (cudaGetSymbolAddress, with that device current) and
 *     caches it; make that first call before any stream capture.
 *   - Every call on a device uses the same array, which keeps what the last
 *     call left there.  Nothing in it needs to start at zero (each call
 *     writes all of H before reading it), but calls whose kernels overlap
 *     on the GPU -- on different streams, or from different host threads --
 *     race on it: order them on one stream or with events.
 */
#define TP_STATIC_WS_BYTES (32u << 20)

tp_status tp_mlp_block_static_ws(const void *X, const void *W1, const void *W2, void *Y,
                                 int64_t M, int64_t d, int64_t f, int n_shards,
                                 tp_dtype in_t, tp_dtype out_t, cudaStream_t s);

/* ------------------------------------------------------------------------
 * Backward pass.  The pages state the structure, not the formulas: the
 * identity operator that feeds every shard the same input in the forward
 * pass becomes an all-reduce -- here an on-device sum over shards -- in the
 * backward pass, and the forward all-reduce becomes an identity: every
 * shard receives the full output gradient (topic page, "Megatron-LM Tensor
 * Parallelism", identity operators); each shard computes the gradients of
 * its own 1/N of the weights (section "Memory Distribution").  For the loss
 * gradient dY = dL/dY of Y = X W the gradients are dW = X^T dY and
 * dX = dY W^T.
 *
 * Conventions as above; bf16 inputs only (TP_ERR_DTYPE otherwise), outputs
 * bf16 (RNE) or fp32 (out_t), K and Nout multiples of 8.  Every gradient is
 * a full dense matrix; a NULL output pointer skips that gradient.  All
 * products run on the tensor cores with fp32 accumulation: X^T and W^T are
 * read in place (the TMA boxes and shared-memory descriptors take the
 * transposed layout), never copied.
 * ---------------------------------------------------------------------- */

/*
 * Backward of tp_column_linear (act = none): X [M,K], W [K,Nout], dY [M,Nout].
 *   dW [K, Nout] = X^T dY   -- column block i of dW is shard i's gradient
 *                              X^T dY_i;
 *   dX [M, K]    = sum_i dY_i W_i^T -- the backward all-reduce, added inside
 *                              the fp32 accumulator in ascending shard order
 *                              (the K loop of dY W^T walks W's columns in
 *                              order).
 * Errors: TP_ERR_DIVISIBILITY if n_shards does not divide Nout.
 */
tp_status tp_column_linear_backward(const void *X, const void *W, const void *dY, void *dX,
                                    void *dW, int64_t M, int64_t K, int64_t Nout, int n_shards,
                                    tp_dtype in_t, tp_dtype out_t, cudaStream_t s);

/*
 * Backward of tp_row_linear: X [M,K], W [K,Nout], dY [M,Nout] (every shard
 * receives the full dY).
 *   dW [K, Nout] = X^T dY   -- row block i of dW is shard i's gradient X_i^T dY;
 *   dX [M, K]    = dY W^T   -- column block i of dX is shard i's dY W_i^T
 *                              (no exchange).
 * The two products are the same as tp_column_linear_backward's; the split
 * only decides which blocks a shard owns.
 * Errors: TP_ERR_DIVISIBILITY if n_shards does not divide K.
 */
tp_status tp_row_linear_backward(const void *X, const void *W, const void *dY, void *dX,
                                 void *dW, int64_t M, int64_t K, int64_t Nout, int n_shards,
                                 tp_dtype in_t, tp_dtype out_t, cudaStream_t s);

/*
 * Bytes of workspace tp_mlp_block_backward needs: three bf16 [M, f] buffers
 * (pre-activation Z, H = GeLU(Z), dZ), each rounded up to 256 bytes.
 * Returns 0 for negative sizes or t other than TP_BF16.
 */
size_t tp_mlp_block_backward_workspace_size(int64_t M, int64_t f, tp_dtype t);

/*
 * Backward of tp_mlp_block for dY [M, d], with the pre-activation recomputed
 * (nothing saved from the forward pass):
 *   Z   = X W1, H = GeLU(Z)        one launch, both stored bf16 (H equals
 *                                  the forward pass's H bit for bit)
 *   dZ  = (dY W2^T) * GeLU'(Z)     GeLU' = Phi + z phi fused into the
 *                                  epilogue, Z read by TMA; stored bf16
 *   dW2 = H^T dY   [f, d]          row block i = shard i
 *   dW1 = X^T dZ   [d, f]          column block i = shard i
 *   dX  = dZ W1^T  [M, d]          shards added in ascending order in the
 *                                  fp32 accumulator (backward all-reduce)
 * ws: at least tp_mlp_block_backward_workspace_size(M, f, in_t) bytes,
 * 16-byte aligned, caller-owned; its contents are not needed afterwards.
 * Any of dX, dW1, dW2 may be NULL.  Errors: as tp_mlp_block.
 */
tp_status tp_mlp_block_backward(const void *X, const void *W1, const void *W2, const void *dY,
                                void *dX, void *dW1, void *dW2, void *ws, size_t ws_bytes,
                                int64_t M, int64_t d, int64_t f, int n_shards, tp_dtype in_t,
                                tp_dtype out_t, cudaStream_t s);

/*
 * Synchronises stream s, then reads and clears the current device's status
 * word.  Returns TP_ERR_DEVICE_TIMEOUT if any kernel of this library gave up
 * a bounded wait since the last call (its outputs are then invalid),
 * TP_ERR_CUDA if the synchronisation failed, TP_OK otherwise.
 */
tp_status tp_get_device_status(cudaStream_t s);

/*
 * Self-test of the bounded-wait machinery: launches one CTA that waits on a
 * shared-memory barrier nobody arrives on, for at most limit_ns nanoseconds
 * (clamped to [1e3, 5e9]), then marks the status word and returns.  After
 * it, tp_get_device_status() must report TP_ERR_DEVICE_TIMEOUT.  The kernel
 * neither faults nor hangs.
 */
tp_status tp_selftest_bounded_wait(uint64_t limit_ns, cudaStream_t s);

/* Human-readable name of a status code (static storage; never NULL). */
const char *tp_status_string(tp_status st);

#ifdef __cplusplus
}
#endif

#endif /* TP_B300_H */

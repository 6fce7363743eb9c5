/*
 * embbwd — backward pass of pooled (EmbeddingBag) and unpooled embedding
 * lookups over many tables, with SGD or row-wise Adagrad applied in place to
 * every unique touched row. GB300 (sm_103a) CUDA kernels behind a plain C ABI.
 *
 * The operation (the problem statement of "fbgemm_gpu/codegen/
 * embedding_backward_split_template.cu", host function
 * split_embedding_backward_codegen_{optimizer}_{weighted}_exact_cuda):
 *
 *   For table t and bag b with lookups i in [offsets[t*B+b], offsets[t*B+b+1]):
 *     G_t[indices[i]] += s_i * grad_output[b, D_offsets[t] : D_offsets[t+1]]
 *   with s_i = per_sample_weights[i] (if given) * (1/L under mean pooling),
 *   L the bag's length. Unpooled ("nobag"): G_t[indices[l]] += grad_output[l, :].
 *   Then, once for every unique touched row (t, idx):
 *     SGD:               w <- w - lr * G
 *     row-wise Adagrad:  m <- m + sum_d(G_d^2)/D_t ;  w <- w - lr * G / (sqrt(m) + eps)
 *   ("tt_embeddings_cuda.cu": update_tt_cores_sgd_kernel and
 *    cache_backward_rowwise_adagrad_approx_kernel give the two update rules;
 *    here they act on the de-duplicated row gradient.)
 *   The update is computed in fp32 and rounded once (round-to-nearest-even,
 *   or stochastically with EMB_FLAG_STOCHASTIC_ROUNDING) to the weight's
 *   storage type. Rows that no lookup touches are not written.
 *
 * Also declared here: elementwise Adagrad (emb_bag_bwd_adagrad), the
 * dense-gradient mode (emb_bag_bwd_dense_grad, emb_nobag_bwd_dense_grad), the
 * forward pooled lookup (emb_bag_fwd), an allocation-free unpooled update
 * (emb_nobag_bwd_sgd_atomic_noalloc), and the exchange step of row-sharded
 * tables over several ranks (emb_shard_*). emb_shard_bucketize is the one call
 * that synchronises (it returns the exchange's split sizes).
 *
 * Layouts (all element offsets, not bytes):
 *   weights        flat; row idx of table t starts at weights_offsets[t] + idx*D_t
 *   momentum       fp32; row idx of table t at momentum_offsets[t] + idx
 *                  (momentum_offsets NULL => hash_size_cumsum[t] + idx)
 *   indices        int64[N], row ids local to their table
 *   offsets        int64[B*T+1], CSR over bags in table-major order (bag t*B+b)
 *   grad_output    pooled: [B, D_offsets[T]] row-major; unpooled: [N, D]
 *   per_sample_weights  fp32[N] or NULL
 *
 * Ownership: every tensor pointer passed to a call is caller-owned device
 * memory. Host arrays given to emb_bwd_plan are copied. The plan owns all of
 * its scratch (device memory sized from max_N at plan time); calls allocate
 * nothing.
 *
 * Execution: calls enqueue work on `stream` (a cudaStream_t; NULL = legacy
 * default stream) and return without synchronising. Argument errors are
 * returned synchronously. Errors found on the device (an index outside its
 * table, malformed offsets, a bounded wait that ran out) are latched in the
 * plan, leave weights and momentum unmodified, and are returned by the next
 * emb_plan_status(). One plan serves one call at a time: calls on one plan
 * must be ordered (same stream, or synchronised), because they share scratch.
 * A call contains no host synchronisation and no allocation, so it can be
 * captured in a CUDA graph.
 */
#ifndef EMBBWD_H
#define EMBBWD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EMB_OK = 0,
  EMB_ERR_INVALID_ARG = 1,         /* bad argument, or malformed offsets found on the device */
  EMB_ERR_UNSUPPORTED = 2,         /* valid but not supported by this library (see each call) */
  EMB_ERR_INDEX_OUT_OF_RANGE = 3,  /* an index outside [0, rows of its table) */
  EMB_ERR_OOM = 4,                 /* plan scratch could not be allocated */
  EMB_ERR_CUDA = 5,                /* a CUDA runtime call failed */
  EMB_ERR_TIMEOUT = 6              /* a bounded inter-block wait ran out; nothing was updated */
} emb_status;

typedef enum { EMB_F32 = 0, EMB_F16 = 1, EMB_BF16 = 2 } emb_dtype;
typedef enum { EMB_POOL_SUM = 0, EMB_POOL_MEAN = 1 } emb_pooling;
typedef enum { EMB_NOBAG_AUTO = 0, EMB_NOBAG_SORTED = 1, EMB_NOBAG_ATOMIC = 2 } emb_nobag_path;

/* emb_bwd_plan flags. Index range checking is always on. */
#define EMB_FLAG_CHECK_INDICES 0x1u
/* Launch the kernels of a call as plain stream-ordered launches instead of
 * programmatic dependent launches (for A/B timing; results are identical). */
#define EMB_FLAG_NO_PDL 0x2u
/* Stochastic rounding of fp16 / bf16 weight stores ("embedding_backward_split_
 * template.cu", the stochastic_rounding argument of the per-row kernels and
 * their Philox-seeded 16-bit stores): an update is rounded to one of its two
 * representable neighbours, away from zero with probability equal to the
 * fraction of an ulp it lies past the one toward zero (unbiased in expectation). Applies to the SGD and Adagrad updates of plans
 * with 16-bit weights (fp32 weights and the dense-gradient mode store as usual).
 * Element d of the row with linear index K, in the update call numbered c, draws
 * word d mod 4 of Philox4x32-10 (Salmon et al., SC 2011) at counter
 * (K, d / 4, c mod 2^32, c / 2^32) under the key (seed mod 2^32, seed / 2^32).
 * bf16: the 16 low bits of the word are added to the fp32 pattern, then it is
 * truncated; fp16: the neighbour away from zero is taken iff (word >> 8) <
 * floor(fraction * 2^24). The call number starts at 0; each SGD or Adagrad
 * call with N > 0 on a plan with 16-bit weights takes the next one;
 * emb_plan_set_rounding sets seed and number.
 * A call captured in a CUDA graph keeps the number it was captured with. */
#define EMB_FLAG_STOCHASTIC_ROUNDING 0x4u
/* Sort with the multi-block front (histogram kernel, radix passes, run-length
 * kernel) even where the small-batch front applies. That front takes calls of
 * at most 2^16 lookups whose tables fit one cluster of CTAs each, all resident
 * at once; a cluster sorts and run-length encodes one table's lookups in
 * shared memory in a single launch. For A/B timing and tests: both fronts
 * give identical results. */
#define EMB_FLAG_NO_CLUSTER_FRONT 0x8u
/* Test only: every block that would wait on another one gives up at once and
 * reports EMB_ERR_TIMEOUT, exercising the error path without a real stall. */
#define EMB_FLAG_DEBUG_FORCE_TIMEOUT 0x100u

typedef struct emb_plan emb_plan;

/* Creates a plan for a fixed set of tables.
 *   device            CUDA device ordinal the plan and all its calls use.
 *   T                 number of tables, 1..4096.
 *   hash_size_cumsum  host int64[T+1]: hash_size_cumsum[t] = rows of tables < t;
 *                     strictly increasing, hash_size_cumsum[0] = 0, total rows < 2^32.
 *                     Row idx of table t has linear index hash_size_cumsum[t] + idx
 *                     ("embedding_backward_split_template.cu", the per-row kernels).
 *   D_offsets         host int32[T+1]: D_t = D_offsets[t+1] - D_offsets[t], each a
 *                     positive multiple of 4 (the pages' vector width) and <= 4096.
 *   weights_offsets   host int64[T], each a multiple of 4.
 *   momentum_offsets  host int64[T] or NULL.
 *   weight_dtype      storage type of weights (fp32, fp16, bf16).
 *   grad_dtype        type of grad_output (fp32, fp16, bf16).
 *   max_N             largest lookup count any call will pass (< 2^30, and
 *                     max_N * ceil(max D_t / 256) < 2^31).
 *   max_B             largest batch any call will pass (max_B * T < 2^31).
 *   max_segment_length_per_warp  runs at least this long take the block-level
 *                     path ("embedding_backward_split_template.cu",
 *                     *_find_long_segments); <= 0 selects 32.
 *   flags             EMB_FLAG_* bits.
 * Returns EMB_ERR_INVALID_ARG for malformed arguments, EMB_ERR_OOM if scratch
 * cannot be allocated, EMB_ERR_CUDA on other runtime failures. *out is NULL on error. */
emb_status emb_bwd_plan(emb_plan** out, int device, int32_t T, const int64_t* hash_size_cumsum,
                        const int32_t* D_offsets, const int64_t* weights_offsets,
                        const int64_t* momentum_offsets, emb_dtype weight_dtype,
                        emb_dtype grad_dtype, int64_t max_N, int32_t max_B,
                        int32_t max_segment_length_per_warp, uint32_t flags);

/* Stochastic rounding state of the plan: `seed` keys the random words and
 * `next_call` is the call number the next update call uses (see
 * EMB_FLAG_STOCHASTIC_ROUNDING). Host-side only; no synchronisation.
 * emb_plan_get_rounding reads both back (either pointer may be NULL). */
emb_status emb_plan_set_rounding(emb_plan* plan, uint64_t seed, uint64_t next_call);
emb_status emb_plan_get_rounding(const emb_plan* plan, uint64_t* seed, uint64_t* next_call);

/* Frees the plan and its scratch (synchronises the device). NULL is accepted. */
emb_status emb_plan_destroy(emb_plan* plan);

/* Pooled backward + SGD, in place on `weights` (plan's weight_dtype).
 * offsets has B*T+1 entries with offsets[0] = 0 and offsets[B*T] = N; B <= max_B,
 * N <= max_N. per_sample_weights may be NULL. N = 0 returns EMB_OK and does nothing
 * ("embedding_backward_split_template.cu": the exact_cuda host function's
 * empty-indices short-circuit and its T > 0, B > 0 checks). */
emb_status emb_bag_bwd_sgd(emb_plan* plan, void* weights, const int64_t* indices,
                           const int64_t* offsets, int64_t N, int32_t B,
                           const float* per_sample_weights, const void* grad_output,
                           emb_pooling mode, float lr, void* stream);

/* Pooled backward + row-wise Adagrad, in place on `weights` and fp32 `momentum`.
 * Same arguments as emb_bag_bwd_sgd plus momentum and eps. Rows of every supported
 * width (D_t <= 4096): when some D_t > 1024 the reduce runs twice on the stream,
 * first finding each row's new state from the sums of squares of its 1024-wide
 * chunks (added in chunk order), then updating the weights. */
emb_status emb_bag_bwd_rowwise_adagrad(emb_plan* plan, void* weights, float* momentum,
                                       const int64_t* indices, const int64_t* offsets,
                                       int64_t N, int32_t B, const float* per_sample_weights,
                                       const void* grad_output, emb_pooling mode, float lr,
                                       float eps, void* stream);

/* Pooled backward + elementwise Adagrad, in place on `weights` and fp32 `momentum`,
 * whose layout is that of the weights (momentum[weights_offsets[t] + idx*D_t + d],
 * 16-byte aligned): for every unique row, with G its de-duplicated gradient,
 *   m_d <- m_d + G_d^2 ;  w_d <- w_d - lr * G_d / (sqrt(m_d) + eps)
 * ("tt_embeddings_cuda.cu", update_tt_cores_adagrad_kernel). Other arguments as
 * for emb_bag_bwd_sgd; rows of any supported width. */
emb_status emb_bag_bwd_adagrad(emb_plan* plan, void* weights, float* momentum,
                               const int64_t* indices, const int64_t* offsets, int64_t N,
                               int32_t B, const float* per_sample_weights,
                               const void* grad_output, emb_pooling mode, float lr, float eps,
                               void* stream);

/* Dense-gradient mode: instead of updating, writes the de-duplicated gradient G of
 * every touched row into `grad_weights`, a buffer of the plan's weight_dtype with
 * the layout of the weights (row idx of table t at grad_weights[weights_offsets[t] +
 * idx*D_t]), after zeroing it over the plan's whole weights extent (the largest
 * weights_offsets[t] + rows_t*D_t), so untouched rows read zero ("embedding_backward_
 * split_template.cu", the dense variant: grad_dev_weights = zeros_like(dev_weights),
 * then grad_sum stored per touched row). G is rounded once to the storage type.
 * Pooled: arguments as for emb_bag_bwd_sgd without lr. Unpooled: as for
 * emb_nobag_bwd_sgd without lr and path (the sorted, deterministic path). */
emb_status emb_bag_bwd_dense_grad(emb_plan* plan, void* grad_weights, const int64_t* indices,
                                  const int64_t* offsets, int64_t N, int32_t B,
                                  const float* per_sample_weights, const void* grad_output,
                                  emb_pooling mode, void* stream);
emb_status emb_nobag_bwd_dense_grad(emb_plan* plan, void* grad_weights, const int64_t* indices,
                                    const int64_t* offsets, int64_t N, int32_t B,
                                    const void* grad_output, void* stream);

/* Unpooled backward + SGD: lookup l adds grad_output[l, :] (shape [N, D], every
 * table has the same D) to row indices[l] of its table, the table given by the
 * CSR offsets (B*T+1 entries; only table membership matters). There is no
 * weighted variant ("embedding_backward_split_template.cu" generates no
 * weighted nobag kernel).
 *   path EMB_NOBAG_SORTED: sort + de-duplicated, deterministic update.
 *   path EMB_NOBAG_ATOMIC: one float atomic add of -lr*g per element, no sort
 *        ("tinygrad/nn/__init__.py", _embedding_bwd_kernel; "tt_embeddings_cuda.cu",
 *        cache_backward_sgd_kernel); fp32 weights only, else EMB_ERR_UNSUPPORTED.
 *   path EMB_NOBAG_AUTO: the faster of the two for the plan's types. */
emb_status emb_nobag_bwd_sgd(emb_plan* plan, void* weights, const int64_t* indices,
                             const int64_t* offsets, int64_t N, int32_t B,
                             const void* grad_output, float lr, emb_nobag_path path,
                             void* stream);

/* Forward pooled lookup (EmbeddingBag forward) over the plan's tables:
 *   output[b, D_offsets[t] + d] = sum over lookups i of bag (t, b) of
 *                                 s_i * weights[weights_offsets[t] + indices[i]*D_t + d],
 *   s_i = per_sample_weights[i] (if not NULL) times 1/L (EMB_POOL_MEAN, L = bag length),
 * the scale the backward applies to the same lookup (the forward is the adjoint
 * of the backward's scatter). "tt_embeddings_cuda.cu", cache_forward_kernel and
 * reduce_output_kernel: a bag's output row is the sum of the rows it indexes.
 *   weights     the plan's weight_dtype, layout as for the backward (read only).
 *   indices, offsets, N, B, per_sample_weights  as for emb_bag_bwd_sgd.
 *   output      [B, D_offsets[T]] of output_dtype (fp32, fp16 or bf16), overwritten
 *               entirely: an empty bag gives zeros; rounded once from fp32 sums.
 * Asynchronous on `stream`; uses no plan scratch, so it may run while no
 * backward call of the plan is in flight on another stream. An index outside its
 * table or malformed offsets latch EMB_ERR_INDEX_OUT_OF_RANGE / EMB_ERR_INVALID_ARG
 * (read with emb_plan_status); the offending lookup or bag is left out. */
emb_status emb_bag_fwd(emb_plan* plan, const void* weights, const int64_t* indices,
                       const int64_t* offsets, int64_t N, int32_t B,
                       const float* per_sample_weights, emb_pooling mode, void* output,
                       emb_dtype output_dtype, void* stream);

/* Allocation-free unpooled atomic SGD (the same update as emb_nobag_bwd_sgd with
 * EMB_NOBAG_ATOMIC), for callers that cannot allocate device memory when they run
 * it: inside a CUDA graph capture, under a runtime that owns all device memory,
 * or where the library must not call the device allocator. The pages have no
 * counterpart of this entry point; it exists for those callers.
 *   No plan is used and nothing is allocated (no cudaMalloc, cudaFree or
 *   allocating library call). Scratch is one fixed static device array in the
 * library image, about 21 KB, present on every GPU that loads the library
 *   until the process exits. Limits: N <= 4194304 lookups, T <= 4096 tables,
 *   B*T < 2^31, D a multiple of 4 and <= 4096; beyond them EMB_ERR_INVALID_ARG.
 *   hash_size_cumsum (int64[T+1]) and weights_offsets (int64[T]) are caller-owned
 *   DEVICE arrays here, checked on the device before any update: hash_size_cumsum
 *   starts at 0, strictly increases and stays below 2^32; every weights_offsets[t]
 *   is >= 0 and a multiple of 4. weights are fp32; grad_output is [N, D] of
 *   grad_dtype. device_status (device uint32, may be NULL) receives this call's
 *   device error bits: 1 = an index outside its table, 2 = malformed offsets,
 *   hash_size_cumsum or weights_offsets; 0 = none. Nothing is updated when a bit
 *   is set.
 *   The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   All calls share the scratch array: calls that overlap on the GPU race, so
 *   order them (one stream, or events). Asynchronous on `stream`. */
emb_status emb_nobag_bwd_sgd_atomic_noalloc(int device, int32_t T,
                                            const int64_t* hash_size_cumsum,
                                            const int64_t* weights_offsets, int32_t D,
                                            float* weights, const int64_t* indices,
                                            const int64_t* offsets, int64_t N, int32_t B,
                                            const void* grad_output, emb_dtype grad_dtype,
                                            float lr, uint32_t* device_status, void* stream);

/* Waits for the plan's last call, then returns and clears the latched device
 * error (EMB_OK if none). */
emb_status emb_plan_status(emb_plan* plan);

/* Host copies of the last sorted call's integer outputs, for parity checks:
 * run_keys (ascending unique linear indices), run_len, cum (exclusive scan of
 * run_len, num_runs+1 entries), num_runs, long_ids (runs with run_len >=
 * max_segment_length_per_warp; the order is unspecified, compare as a set) and
 * num_long. Arrays need `capacity` entries (cum: capacity+1); any pointer may be
 * NULL. Synchronises. EMB_ERR_INVALID_ARG if the last call was not a sorted one or
 * a count exceeds capacity. */
emb_status emb_plan_debug_runs(emb_plan* plan, int64_t capacity, int64_t* run_keys,
                               int32_t* run_len, int32_t* cum, int32_t* num_runs,
                               int32_t* long_ids, int32_t* num_long);

/* Profiling: when enabled, calls record CUDA events between their stages. */
emb_status emb_plan_set_profiling(emb_plan* plan, int enable);

/* Stage durations (ms) of the last profiled call; synchronises. Sorted path:
 * [0] linearise + histogram, [1] radix sort passes, [2] run-length encode and
 * long-run partition (one kernel), [3] 0, [4] reduce + optimizer. Atomic path:
 * [0] index check, [4] atomic scatter, others 0. Writes min(n, 5) values. */
emb_status emb_plan_stage_ms(emb_plan* plan, float* ms, int32_t n);

/* ---- Row-wise sharding over W ranks (the exchange step before the backward).
 * Every rank trains on its own batch and owns a contiguous row range of every
 * table: rank r holds rows [row_bounds[t*(W+1)+r], row_bounds[t*(W+1)+r+1]) of
 * table t, the vocabulary sharding of "Function _embedding_bwd_kernel" (tinygrad:
 * a device owns one slice of the rows; lookups outside it add nothing there).
 * A step on rank r:
 *   1. emb_shard_bucketize its batch: per owner, the lookups of its rows;
 *   2. all-to-all the parts (offsets: W*(T*B+1) each way; indices and scales
 *      with the per-owner counts as split sizes) and all-gather grad_output into
 *      [W*B, sum D] in rank order (e.g. NCCL through torch.distributed);
 *   3. emb_shard_merge the received parts into one batch of W*B bags per table;
 *   4. the ordinary backward on the rank's own plan (its local tables: row range
 *      sizes as hash_size_cumsum, rows relative to the range) with B' = W*B, the
 *      merged offsets and indices, the merged scales as per_sample_weights (or
 *      NULL when the batch is unweighted and sum-pooled) and EMB_POOL_SUM.
 * The forward runs 1-3 the same way, then emb_bag_fwd with B' = W*B gives the
 * rank's partial sums of every rank's bags, and a reduce-scatter over ranks
 * gives each rank its own bags' output. */
typedef struct emb_shard emb_shard;

/* Creates the shard map of one rank: T tables (1..4096), W ranks (1..256),
 * row_bounds host int64[T*(W+1)] (row_bounds[t*(W+1)] = 0, non-decreasing, last
 * = rows of table t > 0; empty ranges are allowed here, but a rank whose plan
 * has an empty table cannot create that plan), max_B the largest per-rank batch
 * (W * T * max_B < 2^31). Allocates its scratch on `device` (about
 * 12 * W * T * max_B bytes). */
emb_status emb_shard_create(emb_shard** out, int device, int32_t T, int32_t W,
                            const int64_t* row_bounds, int32_t max_B);

/* The cyclic map: rank r owns rows r, r + W, r + 2W, ... of every table (its
 * local row k is row k*W + r), so a skewed id distribution spreads over all
 * ranks. rows: host int64[T], each > 0. Rows are then relative as row / W in
 * send_indices; a rank's plan has ceil((rows_t - r) / W) rows of table t. */
emb_status emb_shard_create_cyclic(emb_shard** out, int device, int32_t T, int32_t W,
                                   const int64_t* rows, int32_t max_B);
emb_status emb_shard_destroy(emb_shard* shard);

/* Step 1 on `stream`; synchronises it (the exchange needs the sizes on the
 * host). Inputs as for emb_bag_bwd_sgd (device indices [N], offsets [T*B+1],
 * optional per_sample_weights [N], mode). Outputs (device, caller-owned):
 *   send_offsets int64[W][T*B+1]: owner r's bag offsets counted from its first lookup;
 *   send_indices int64[N]: owner 0's lookups first, then owner 1's, ..., each row
 *     relative to the owner's range (cyclic map: row / W), in bag order and
 *     lookup order within a bag;
 *   send_scales float[N] or NULL: per-sample weight (1 if none), divided in fp32
 *     by the length of its whole bag under mean pooling;
 *   send_counts host int64[W]: lookups per owner (the all-to-all split sizes).
 * EMB_ERR_INDEX_OUT_OF_RANGE for an index outside its table, EMB_ERR_INVALID_ARG
 * for malformed offsets; nothing usable is written then. */
emb_status emb_shard_bucketize(emb_shard* shard, const int64_t* indices, const int64_t* offsets,
                               int64_t N, int32_t B, const float* per_sample_weights,
                               emb_pooling mode, int64_t* send_offsets, int64_t* send_indices,
                               float* send_scales, int64_t* send_counts, void* stream);

/* Step 3 on `stream`, asynchronous. recv_offsets device int64[W][T*B+1] (source
 * s's send_offsets for this rank, in source order), recv_indices / recv_scales
 * the n_recv received lookups concatenated in source order (recv_scales may be
 * NULL, then merged_scales must be NULL too). Writes merged_offsets int64[T*W*B+1]
 * and merged_indices / merged_scales [n_recv]: bag s*B + b of table t holds
 * source s's bag (t, b). Received offsets inconsistent with n_recv are skipped
 * and reported by emb_shard_status as EMB_ERR_INVALID_ARG. */
emb_status emb_shard_merge(emb_shard* shard, const int64_t* recv_offsets, const int64_t* recv_indices,
                           const float* recv_scales, int64_t n_recv, int32_t B,
                           int64_t* merged_offsets, int64_t* merged_indices, float* merged_scales,
                           void* stream);

/* Waits for the shard's last call and returns (and clears) its latched errors. */
emb_status emb_shard_status(emb_shard* shard);

/* Static description of a status code. */
const char* emb_status_string(emb_status status);

#ifdef __cplusplus
}
#endif

#endif /* EMBBWD_H */

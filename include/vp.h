/*
 * vp.h -- C ABI of libvp: vocab-parallel cross-entropy over a tied,
 * vocab-sharded LM head, and the vocab-sharded embedding gather, on one
 * B300 (sm_103a).
 *
 * Notation: N tokens, H hidden size, V vocabulary size, T vocab shards.
 * X is [N,H] row-major, W is [V,H] row-major and tied between the embedding
 * and the LM head.  Shard t owns vocab ids [t*V/T, (t+1)*V/T)  (MiniMind-tron
 * book, ch. 5 "Vocab Parallelism", sec. 5.1 and 5.2.1); V % T must be 0.
 * On one GPU the T shards are a tiling of the vocab dimension inside the
 * kernels and every cross-shard reduction the pages do with a collective is
 * an on-device reduction; nothing here talks to another GPU.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers owned by the caller (the library keeps no
 *     reference after the call returns); the library never allocates device
 *     memory -- scratch comes from the caller's `workspace`.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).  A returned VP_OK means "arguments
 *     accepted and kernels launched"; results are ready when the stream is.
 *   - dtype applies to X, W, the embedding output and dX.  VP_BF16 runs on the
 *     tcgen05 tensor cores with fp32 accumulation; VP_F32 runs on CUDA-core
 *     FMAs (no TF32) for full fp32 accuracy.
 *   - Arguments are checked before any launch: N, H, V, T <= 0 or V % T != 0
 *     -> VP_ERR_INVALID_ARG; a NULL required pointer -> VP_ERR_INVALID_ARG;
 *     a pointer not 16-byte aligned, H*sizeof(dtype) not a multiple of 16,
 *     or a GEMM with 2^31 or more 128x256 output tiles (N*V, V*H or N*H
 *     beyond about 7e13) -> VP_ERR_UNSUPPORTED; a workspace smaller than the minimum
 *     -> VP_ERR_WORKSPACE; a CUDA launch error -> VP_ERR_CUDA.  On any error
 *     nothing has been launched or written, except for VP_ERR_CUDA.
 *   - Every wait inside a kernel is bounded in time.  A wait that runs out
 *     sets a bit in the workspace's device status word (vp_read_device_status)
 *     and the kernel returns early; outputs are then undefined, and a forward
 *     whose GEMM gave up writes NaN to loss, lse and the shard statistics.
 */
#ifndef VP_H
#define VP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { VP_F32 = 0, VP_BF16 = 1 } vp_dtype;

typedef enum {
  VP_OK = 0,
  VP_ERR_INVALID_ARG = 1,
  VP_ERR_UNSUPPORTED = 2,
  VP_ERR_WORKSPACE = 3,
  VP_ERR_CUDA = 4
} vp_status;

/* Device status bits written into the workspace header by the kernels. */
#define VP_DEV_TIMEOUT_PRODUCER 0x1u /* TMA producer gave up waiting for a free stage  */
#define VP_DEV_TIMEOUT_MMA      0x2u /* MMA issuer gave up waiting for data / TMEM      */
#define VP_DEV_TIMEOUT_EPILOGUE 0x4u /* epilogue gave up waiting for an accumulator     */

/* Human-readable name of a status code (static storage). */
const char* vp_status_string(vp_status s);

/* Library version string, e.g. "libvp 0.1 sm_103a". */
const char* vp_version(void);

/*
 * vp_embed_fwd -- vocab-parallel embedding lookup, the shard outputs summed.
 *
 * "Vocab Parallelism" sec. 5.2.1 (masked local lookup; the V=8 worked table)
 * and "Vocab parallelism: how to split embedding and LM head", figure 1:
 * shard t maps an id outside [t*V/T,(t+1)*V/T) to local row 0, looks it up
 * and zeroes the row; the T shard outputs are summed.  Exactly one shard
 * contributes, so
 *     out[n,:] = +0.0 + W[ids[n],:]   if 0 <= ids[n] < V
 *     out[n,:] = 0                    otherwise,
 * bit-exact (a -0.0 weight comes out +0.0, as a sum from +0.0 gives).
 *
 *   ids  int64 [N]        token ids (any value; out-of-range ids give zero rows)
 *   W    dtype [V,H]      tied weight, row-major
 *   out  dtype [N,H]      written, row-major
 * Requires H*sizeof(dtype) % 16 == 0 and 16-byte aligned W and out.
 */
vp_status vp_embed_fwd(const int64_t* ids, const void* W, void* out,
                       int64_t N, int64_t H, int64_t V, int T, vp_dtype dtype,
                       void* stream);

/*
 * vp_embed_fwd_sp -- vp_embed_fwd with sequence parallelism on: one rank's
 * slice of the reduce-scattered shard sum.
 *
 * "Vocab Parallelism" sec. 5.2.1: with SP off the T shard outputs are
 * all-reduced (vp_embed_fwd); with SP on they are reduce-scattered along the
 * token dimension, so rank r keeps token rows [r*N/T, (r+1)*N/T) of the sum:
 *     out[i,:] = vp_embed_fwd(ids, W)[rank*N/T + i, :],   i < N/T
 * bit-exact, same -0.0 rule.  The T ranks' outputs stacked in rank order are
 * the SP-off output.  Its backward (the all-gather of the ranks' upstream
 * slices, then each shard's masked scatter) is vp_embed_bwd on the stacked
 * [N,H] upstream gradient.
 *
 *   ids   int64 [N]        all N token ids (rank r reads its N/T)
 *   W     dtype [V,H]
 *   out   dtype [N/T,H]    written
 *   rank  0 <= rank < T;  N % T must be 0 (else VP_ERR_INVALID_ARG)
 */
vp_status vp_embed_fwd_sp(const int64_t* ids, const void* W, void* out,
                          int64_t N, int64_t H, int64_t V, int T, int rank,
                          vp_dtype dtype, void* stream);

/*
 * vp_embed_bwd -- backward of vp_embed_fwd into the tied weight's gradient.
 *
 * "Vocab Parallelism" sec. 5.2.1: shard t's lookup zeroes the output rows of
 * ids outside its range, so those rows pass it no gradient, and the gather
 * adds every other token's upstream row into local row id - t*V/T.  Summed
 * over the shards (each sees the same upstream rows, the forward's sum being
 * an all-reduce), weight row v receives the rows of exactly the tokens with
 * id v.  Sec. 5.2.2 ties the embedding and the LM head to one parameter, so
 * its gradient is the sum of both layers': pass the LM head's dW (from
 * vp_lmhead_ce_bwd or vp_lmhead_ce_fwd_bwd) with accumulate = 1.
 *     dW[v,:] = (accumulate ? dW[v,:] : 0) + sum_{n: ids[n] = v} dOut[n,:]
 * in fp32; ids outside [0,V) contribute nothing.  Deterministic: no atomics;
 * each row's sum runs over its tokens in increasing n in runs of 32 sorted
 * positions, the run sums added in order, then added to the existing row.
 *
 *   ids       int64 [N]
 *   dOut      dtype [N,H]    upstream gradient of the embedding output
 *   dW        f32 [V,H]      accumulate != 0: added to; 0: overwritten
 *                            (rows no token names are set to zero)
 *   workspace >= vp_embed_bwd_workspace_size(N, H, V, T, dtype) bytes,
 *             16-byte aligned (sort keys and per-run partial sums)
 * Requires H*sizeof(dtype) % 16 == 0 and 16-byte aligned dOut, dW.
 */
size_t vp_embed_bwd_workspace_size(int64_t N, int64_t H, int64_t V, int T, vp_dtype dtype);
vp_status vp_embed_bwd(const int64_t* ids, const void* dOut, float* dW,
                       int64_t N, int64_t H, int64_t V, int T, vp_dtype dtype,
                       int accumulate, void* workspace, size_t ws_bytes, void* stream);

/*
 * vp_embed_bwd_plan / vp_embed_bwd_planned -- vp_embed_bwd in two steps.
 * The grouping of the tokens by id (a sort of the (id, n) keys, latency-bound
 * index work) needs only the ids, which a training step knows from its start;
 * the sums need dOut.  vp_embed_bwd_plan sorts into `workspace`, for instance
 * on a side stream while the LM head runs; vp_embed_bwd_planned, later, adds
 * the rows into dW from that workspace (same N, H, V, T; the workspace left
 * untouched in between).  Together they compute what vp_embed_bwd computes,
 * bit for bit.  Arguments and errors as for vp_embed_bwd.
 */
vp_status vp_embed_bwd_plan(const int64_t* ids, int64_t N, int64_t H, int64_t V, int T,
                            void* workspace, size_t ws_bytes, void* stream);
vp_status vp_embed_bwd_planned(const void* dOut, float* dW, int64_t N, int64_t H, int64_t V, int T,
                               vp_dtype dtype, int accumulate, void* workspace, size_t ws_bytes,
                               void* stream);

/*
 * vp_lmhead_ce_workspace_size -- bytes of device workspace for a call.
 *   pass 0: vp_lmhead_ce_fwd (exact size needed).
 *   pass 1: vp_lmhead_ce_bwd with the vocab processed in chunks of
 *           `vocab_chunk` ids (<= 0 or >= V: one chunk, the fastest).  Any
 *           workspace at least this large for some chunk works; the backward
 *           derives its chunk from the bytes it is given.
 *   pass 3: the `saved` buffer of vp_lmhead_ce_fwd_keep / vp_lmhead_ce_bwd_saved
 *           (VP_BF16: about N * (2*round8(V) + 20*V/256) bytes, all N tokens;
 *           VP_F32: as pass 2).
 *   pass 2: vp_lmhead_ce_fwd_bwd.  VP_BF16: the last argument is a TOKEN
 *           chunk (rounded down to a multiple of 128; <= 0 or >= N: all N
 *           tokens at once, the fastest), about N_c * (2*round8(V) + 20*V/256)
 *           bytes; the call derives its chunk from the bytes it is given.
 *           VP_F32: the larger of pass 0 and pass 1 (last argument = vocab chunk).
 * Returns 0 for invalid arguments.
 */
size_t vp_lmhead_ce_workspace_size(int64_t N, int64_t H, int64_t V, int T,
                                   vp_dtype dtype, int pass, int64_t vocab_chunk);

/*
 * vp_lmhead_ce_fwd -- fused LM head + vocab-parallel cross-entropy, forward.
 *
 * "Vocab Parallelism" sec. 5.3.1 and the interview note's figure 2 / key
 * formulas: Z = X W^T is produced tile by tile and never stored.  For every
 * shard t and token n the kernel reduces its logits slice to the local max
 * m_t, the local sum S_t = sum exp(z - m_t) and the local target logit
 * z_y^(t) (0 off-shard); an on-device merge gives
 *     m = max_t m_t,  S = sum_t S_t e^(m_t - m),  lse = m + log S,
 *     loss[n] = log S - (z_y - m)              (0 for ignored targets),
 *     loss_mean = sum_n loss[n] / max(1, N_valid)   (sec. 5.3.3).
 * S is carried as S = 1 + R, R the sum without one maximal term, and the loss
 * is formed as log1p(R) + (m - z_y): two non-negative terms, so a loss far
 * below lse (the target is the row's maximum by a wide margin) keeps its
 * relative accuracy instead of cancelling.
 * A target equal to ignore_index, or outside [0,V), is ignored; the latter
 * kind is counted in n_bad.
 *
 *   X         dtype [N,H]    hidden states
 *   W         dtype [V,H]    tied weight
 *   targets   int64 [N]
 *   loss      f32 [N]        written
 *   lse       f32 [N]        written (log-sum-exp of every row, ignored or not;
 *                            the backward consumes it)
 *   loss_mean f32 [1]        written, or NULL
 *   shard_stats f32 [T][3][N] written as (m_t, S_t, z_y^(t)), or NULL
 *   n_bad     int32 [1]      written, or NULL
 *   workspace device bytes >= vp_lmhead_ce_workspace_size(..., pass 0, 0),
 *             16-byte aligned; overwritten.
 */
vp_status vp_lmhead_ce_fwd(const void* X, const void* W, const int64_t* targets,
                           int64_t N, int64_t H, int64_t V, int T,
                           int64_t ignore_index, vp_dtype dtype,
                           float* loss, float* lse, float* loss_mean,
                           float* shard_stats, int32_t* n_bad,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * vp_lmhead_ce_fwd_noalloc -- vp_lmhead_ce_fwd for callers that cannot
 * allocate device memory.  The source pages have no counterpart to this call;
 * it exists for users of this library.
 *
 * Some callers have no device allocator to draw a workspace from: a plugin
 * whose host hands it only input and output buffers, or a latency-bound loop
 * that must never call cudaMalloc (which can synchronise the device and has
 * no time bound).  This call takes the same inputs and outputs as
 * vp_lmhead_ce_fwd and computes the same results, but keeps its scratch in a
 * fixed 32 MiB device array inside libvp instead of a caller workspace.
 *
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - Every GPU that loads libvp holds the 32 MiB array until the process exits.
 *   - Size limit: 256 + ceil(V/tile)*slots*N*8 + N*4 bytes (rounded up to 256)
 *     must fit in 32 MiB, where tile = 256 (bf16) or 64 (f32) and slots is the
 *     number of shard segments one tile can touch (2 when V/T >= tile, at most
 *     T).  Larger sizes return VP_ERR_WORKSPACE and launch nothing.  Example:
 *     N=4096, V=6400, T=2, bf16 needs 1.6 MiB; N=16384, V=128256 does not fit.
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Calls whose executions overlap on the GPU (different streams, or
 *     different host threads on one device) race on it: serialise them.
 *   - The device status word lives in the shared array and is not readable
 *     through vp_read_device_status; if a kernel gives up a wait, loss, lse,
 *     loss_mean and shard_stats come out NaN instead.
 *   - The array's device address is looked up on a device's first successful
 *     call and kept; cudaDeviceReset unloads the library's device code, so do
 *     not call this function on a device after resetting it in this process.
 */
vp_status vp_lmhead_ce_fwd_noalloc(const void* X, const void* W, const int64_t* targets,
                                   int64_t N, int64_t H, int64_t V, int T,
                                   int64_t ignore_index, vp_dtype dtype,
                                   float* loss, float* lse, float* loss_mean,
                                   float* shard_stats, int32_t* n_bad, void* stream);

/*
 * vp_lmhead_ce_bwd -- backward of vp_lmhead_ce_fwd.
 *
 * "Vocab Parallelism" sec. 5.3.2 and the interview note's key formulas: the
 * logit gradient is local to each shard, dZ[n,j] = g_n (softmax_j - 1[j=y_n]),
 * with g_n = dloss[n], or, when dloss is NULL, dmean[0]/max(1,N_valid) (the
 * gradient of dmean * loss_mean; dmean NULL means 1), on valid tokens and 0 on
 * ignored ones.  Each logit tile is
 * recomputed from X and W, dZ is formed in the epilogue and stored in bf16
 * (f32 for VP_F32) scratch for one vocab chunk, then
 *     dW[chunk] = dZ_chunk^T X,     dX += dZ_chunk W[chunk]
 * run on the tensor cores; the sum of dX over chunks is the on-device form of
 * the column-parallel LM head's dX all-reduce.
 *
 *   lse    f32 [N]           from vp_lmhead_ce_fwd
 *   dloss  f32 [N] or NULL
 *   dmean  f32 [1] (device) or NULL: upstream gradient of loss_mean, used
 *          when dloss is NULL (autograd's incoming gradient, a loss scale)
 *   dX     dtype [N,H]       overwritten
 *   dW     f32 [V,H]         overwritten (fp32 so that a caller can add the
 *                            tied embedding's gradient)
 *   workspace  >= vp_lmhead_ce_workspace_size(..., pass 1, c) for some chunk c
 */
vp_status vp_lmhead_ce_bwd(const void* X, const void* W, const int64_t* targets,
                           const float* lse, const float* dloss, const float* dmean,
                           int64_t N, int64_t H, int64_t V, int T,
                           int64_t ignore_index, vp_dtype dtype,
                           void* dX, float* dW,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * vp_lmhead_ce_fwd_bwd -- forward and backward in one call, with the
 * probabilities saved in between instead of recomputed.
 *
 * "Vocab Parallelism" sec. 5.3.1-5.3.3: the forward of vp_lmhead_ce_fwd and
 * the backward of vp_lmhead_ce_bwd for an upstream gradient known up front
 * (dloss, or the mean over valid tokens when dloss is NULL, the usual
 * training case).  Sec. 5.3.2 keeps each shard's softmax from the forward for
 * its local gradient p - onehot; here the forward's epilogue writes, for every
 * 256-wide vocab tile, p = exp(z - m_tile) in fp16 (m_tile = the row's maximum
 * over that tile) next to the (m_t, S_t, z_y^(t)) statistics, the merge gives
 * lse, one bandwidth-bound pass turns p in place into
 *     dZ = g (p exp(m_tile - lse) - 1[j=y])   (bf16),
 * and dW = dZ^T X, dX = dZ W run on the tensor cores.  Against
 * vp_lmhead_ce_fwd + vp_lmhead_ce_bwd this skips the logit recompute
 * (6NHV instead of 8NHV flops) at the price of holding N_c x V 2-byte
 * probabilities: tokens are processed in chunks of N_c rows (all N when the
 * workspace allows), so the fp32 [N,V] logits are never materialised and the
 * saved tile is bounded by the workspace.  The f32 dtype runs the forward and
 * the recompute backward of the split calls.
 *
 * Arguments and outputs are those of vp_lmhead_ce_fwd and vp_lmhead_ce_bwd:
 *   dloss      f32 [N] or NULL (NULL: gradient of dmean * loss_mean)
 *   dmean      f32 [1] (device) or NULL (= 1), used when dloss is NULL
 *   loss, lse  f32 [N] written;  loss_mean, shard_stats, n_bad as in the forward
 *   dX         dtype [N,H] overwritten;  dW  f32 [V,H] overwritten
 *   workspace  >= vp_lmhead_ce_workspace_size(..., pass 2, c) for some chunk c
 * Errors as for the other calls; nothing is launched on an argument error.
 */
vp_status vp_lmhead_ce_fwd_bwd(const void* X, const void* W, const int64_t* targets,
                               const float* dloss, const float* dmean,
                               int64_t N, int64_t H, int64_t V, int T,
                               int64_t ignore_index, vp_dtype dtype,
                               float* loss, float* lse, float* loss_mean,
                               float* shard_stats, int32_t* n_bad,
                               void* dX, float* dW,
                               void* workspace, size_t ws_bytes, void* stream);

/*
 * vp_lmhead_ce_fwd_keep / vp_lmhead_ce_bwd_saved -- the forward and backward
 * of vp_lmhead_ce_fwd_bwd as two calls, for when the upstream gradient is
 * only known later (an autograd backward).
 *
 * "Vocab Parallelism" sec. 5.3.2 saves each shard's softmax in the forward
 * for the local p - onehot of the backward.  vp_lmhead_ce_fwd_keep computes
 * what vp_lmhead_ce_fwd computes (same kernels, same bits) and leaves, in the
 * caller's `saved` buffer, p = exp(z - m_tile) in fp16 and the tile maxima
 * m_tile of every 256-wide vocab tile.  vp_lmhead_ce_bwd_saved then forms
 * c = g exp(m_tile - lse), dZ = c p - g 1[j=y] in place and runs dW = dZ^T X,
 * dX = dZ W: 6NHV flops in all, as in the one-call form, against 8NHV for
 * vp_lmhead_ce_fwd + vp_lmhead_ce_bwd.  The results equal vp_lmhead_ce_fwd_bwd's
 * bit for bit.
 *
 *   saved  device buffer >= vp_lmhead_ce_workspace_size(..., pass 3, 0) bytes,
 *          16-byte aligned, owned by the caller; it must stay untouched from
 *          the forward to the backward, and the backward consumes it (one
 *          backward per forward).
 *   the other arguments as in vp_lmhead_ce_fwd and vp_lmhead_ce_bwd (lse
 *   from the forward; dloss / dmean the upstream gradient).
 * VP_F32 runs vp_lmhead_ce_fwd and the recompute backward in `saved`.
 */
vp_status vp_lmhead_ce_fwd_keep(const void* X, const void* W, const int64_t* targets,
                                int64_t N, int64_t H, int64_t V, int T,
                                int64_t ignore_index, vp_dtype dtype,
                                float* loss, float* lse, float* loss_mean,
                                float* shard_stats, int32_t* n_bad,
                                void* saved, size_t saved_bytes, void* stream);
vp_status vp_lmhead_ce_bwd_saved(const void* X, const void* W, const int64_t* targets,
                                 const float* lse, const float* dloss, const float* dmean,
                                 int64_t N, int64_t H, int64_t V, int T,
                                 int64_t ignore_index, vp_dtype dtype,
                                 void* dX, float* dW,
                                 void* saved, size_t saved_bytes, void* stream);

/*
 * One shard per rank: the building blocks of the T-GPU form.
 *
 * "Vocab Parallelism" sec. 5.3.1 and the interview note's figure 2: each of T
 * ranks holds only its shard W_t = W[t*V/T, (t+1)*V/T) and computes, for every
 * token, three scalars of its logits slice; three all-reduces of [B,S]
 * tensors (MAX, SUM, SUM) combine them.  Sec. 5.3.2 and the key formulas: the
 * logit gradient is local to each rank, dW_t stays local, and the LM head's dX
 * is all-reduced over ranks.  A rank runs
 *     vp_lmhead_ce_shard_fwd  -> stats_t [3][N]
 *     (all-gather of stats_t over the T ranks: [T][3][N]; the caller's collective)
 *     vp_lmhead_ce_merge_stats -> loss, lse (every rank the same)
 *     vp_lmhead_ce_shard_bwd  -> dX_t (fp32), dW_t
 *     (all-reduce SUM of dX_t over the ranks: dX; the caller's collective)
 * One all-gather of 3 floats per token replaces the three all-reduces (m_t is
 * kept local, so the sums need no second round).  On one GPU these calls run
 * the ranks one after another; the library itself never talks to another GPU.
 *
 * vp_lmhead_ce_shard_fwd -- shard t's statistics.
 *   X        dtype [N,H];   W_t  dtype [V/T,H], the shard's rows of the weight
 *   targets  int64 [N]      ids of the whole vocabulary [0,V)
 *   stats    f32 [3][N]     written: m_t (the shard's max logit), R_t = S_t - 1
 *                           (sum of exp(z - m_t) over the shard except one
 *                           maximal term, kept apart from the 1 for accuracy),
 *                           z_y^(t) (the target logit if the valid target lies
 *                           in the shard, else 0)
 *   workspace >= vp_lmhead_ce_workspace_size(N, H, V/T, 1, dtype, 0, 0) bytes
 *   0 <= t < T, V % T == 0 (else VP_ERR_INVALID_ARG); other rules as vp_lmhead_ce_fwd.
 *
 * vp_lmhead_ce_merge_stats -- the merge of the gathered statistics.
 *   stats    f32 [T][3][N]  shard t's stats_t at [t] (device memory)
 *   writes loss [N], lse [N] as vp_lmhead_ce_fwd does (m = max_t m_t,
 *   1 + R = sum_t (1 + R_t) e^(m_t - m), z_y = sum_t z_y^(t),
 *   loss = log1p(R) + (m - z_y), lse = m + log1p(R)), and loss_mean / n_bad
 *   when not NULL.
 *
 * vp_lmhead_ce_shard_bwd -- shard t's backward, recomputing its logits.
 *   lse      f32 [N]        from vp_lmhead_ce_merge_stats
 *   dloss / dmean           as in vp_lmhead_ce_bwd (N_valid counts the whole batch)
 *   dX_t     f32 [N,H]      overwritten: dZ_t W_t, this shard's part of dX (sum
 *                           over t, then round to the training dtype)
 *   dW_t     f32 [V/T,H]    overwritten: dZ_t^T X, complete for the shard
 *   workspace >= vp_lmhead_ce_workspace_size(N, H, V/T, 1, dtype, 1, chunk)
 *             for some vocab chunk (the call derives it from the bytes)
 */
vp_status vp_lmhead_ce_shard_fwd(const void* X, const void* W_t, const int64_t* targets,
                                 int64_t N, int64_t H, int64_t V, int T, int t,
                                 int64_t ignore_index, vp_dtype dtype, float* stats,
                                 void* workspace, size_t ws_bytes, void* stream);
vp_status vp_lmhead_ce_merge_stats(const float* stats, const int64_t* targets,
                                   int64_t N, int64_t V, int T, int64_t ignore_index,
                                   float* loss, float* lse, float* loss_mean, int32_t* n_bad,
                                   void* stream);
vp_status vp_lmhead_ce_shard_bwd(const void* X, const void* W_t, const int64_t* targets,
                                 const float* lse, const float* dloss, const float* dmean,
                                 int64_t N, int64_t H, int64_t V, int T, int t,
                                 int64_t ignore_index, vp_dtype dtype,
                                 float* dX_t, float* dW_t,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * vp_read_device_status -- synchronise `stream` and copy the device status
 * word of `workspace` (VP_DEV_* bits; 0 = no kernel gave up waiting) into
 * *flags.  The word is cleared at the start of every fwd/bwd call.
 */
vp_status vp_read_device_status(const void* workspace, uint32_t* flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VP_H */

/*
 * ttt.h -- C ABI of libttt: the TTT-E2E inner-loop (test-time training) prefill
 * on one B300 GPU.
 *
 * The operation (pages "把 Transformer 做成“终身学习者”：TTT-E2E 如何让大模型边用边学？",
 * §4.2 "推理阶段（Inner Loop 复用）" and §4.4 "伪代码"; "TTT-E2E技术：突破大语言模型上下文限制的新范式",
 * §2.1 "参数更新机制"): text is fed chunk by chunk; for each chunk of at most b
 * tokens a decoder-only Transformer with sliding-window attention (window k,
 * k >= b) runs forward, the mean next-token cross-entropy over the chunk is
 * taken, the loss is backpropagated through the last quarter of the blocks
 * only, and one SGD step W <- W - eta*dW is applied to the MLP weights
 * (W_up, W_down) of those blocks -- the "fast weights" -- before the next chunk.
 * The key/value cache keeps only the last k positions per layer.
 *
 * Model: pre-norm blocks h = x + Attn(RMSNorm(x)), y = h + GELU_tanh(RMSNorm(h).W_up).W_down,
 * logits = RMSNorm(x_L).W_lm; multi-head attention with rotate-half RoPE
 * (inv_freq_i = theta^(-2i/d_head), absolute positions from 0), scale
 * 1/sqrt(d_head), query p sees keys j with p - k < j <= p; no biases.
 *
 * Ownership: the context owns all device memory.  Host pointers passed in are
 * read or written only during the call and never retained.
 * Streams: all work is ordered on the stream given to ttt_create.  Inside a
 * call the context may fork work onto streams of its own (side streams of one
 * sequence; one lane of streams per sequence, up to 4 sequences at a time) and
 * joins them back into that stream before the call returns, so later work on
 * the given stream sees every result.
 * Devices and threads: one process drives one GPU.  The library caches launch
 * settings (per-kernel shared-memory limits, the SM count) on first use, so
 * every context of a process must live on the same device, and calls that
 * launch work must not run concurrently from several host threads.
 * Errors: every call returns 0 or a negative TTT_ERR_* code; after an error the
 * context may only be reloaded (ttt_load_weights) or destroyed.
 */
#ifndef TTT_H
#define TTT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TTT_API __attribute__((visibility("default")))
#else
#define TTT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define TTT_OK 0
#define TTT_ERR_ARG (-1)         /* null pointer, n outside 1..b, token id outside [0, vocab), k < b, ... */
#define TTT_ERR_UNSUPPORTED (-2) /* a shape the library does not handle (see ttt_create)                */
#define TTT_ERR_STATE (-3)       /* prefill before ttt_load_weights                                     */
#define TTT_ERR_OOM (-4)         /* device allocation failed                                            */
#define TTT_ERR_CUDA (-5)        /* a CUDA runtime call failed                                          */
#define TTT_ERR_DEVICE (-6)      /* a kernel reported an error: bounded wait expired or bad token id    */

typedef struct ttt_ctx ttt_ctx;

typedef struct {
  int32_t n_layers;     /* L                                                        */
  int32_t n_trainable;  /* S = number of trailing blocks whose MLPs learn; L/4       */
  int32_t d_model;      /* d                                                        */
  int32_t n_heads;      /* H; d_head = d / H                                        */
  int32_t d_ff;         /* MLP hidden width (4d in every shipped workload)          */
  int32_t vocab;        /* V                                                        */
  int32_t window;       /* k: a query sees the k most recent positions, itself included */
  int32_t chunk;        /* b: tokens per inner-loop step, k >= b                    */
  int32_t n_seqs;       /* independent sequences, each with its own fast weights and cache */
  double rope_theta;
  float rms_eps;        /* 1e-6 */
  float eta;            /* SGD step size of the inner loop */
  int32_t compute;      /* 0: fp32 (every product as three bf16 products of hi/lo
                           halves, fp32 accumulate); 1: bf16 operands, fp32
                           accumulate; fast weights are fp32 in both           */
  int32_t dual_mlp;     /* 0: one MLP per block.  1: the dual-MLP variant ("从KV Cache到
                           权重压缩：大模型持续学习的新范式", §2.2): each trainable block
                           adds a frozen static MLP on the same normalised input,
                           y = h + GELU(n.W_up).W_down + GELU(n.W_up_s).W_down_s,
                           n = RMSNorm(h); only W_up, W_down are fast weights   */
} ttt_config;

/*
 * Create a context on the current CUDA device; work goes to `cuda_stream`
 * (cudaStream_t, NULL = default stream).
 * Supported: d_head % 16 == 0 and d_head <= 128 (<= 64 when compute == 0),
 * d_model % 64 == 0, d_model <= 4096, d_ff % 64 == 0, vocab % 8 == 0, window % 128 == 0,
 * 1 <= chunk <= window, 1 <= n_trainable <= n_layers.  Otherwise
 * TTT_ERR_UNSUPPORTED (shape) or TTT_ERR_ARG (inconsistent values).
 */
TTT_API int ttt_create(const ttt_config* cfg, void* cuda_stream, ttt_ctx** out);

/*
 * Copy the fp32 weight blob (host memory, n_floats values) to the device and
 * reset every sequence: position 0, empty cache, fast weights = the loaded
 * W_up / W_down of the trainable blocks.  Blob order, all row-major, y = x.W:
 *   E[V][d];
 *   for each layer: g_attn[d], Wq[d][d], Wk[d][d], Wv[d][d], Wo[d][d],
 *                   g_mlp[d], W_up[d][d_ff], W_down[d_ff][d];
 *   g_final[d]; W_lm[d][V].
 * With dual_mlp = 1, each trainable layer (the last n_trainable) adds its
 * static pair W_up_s[d][d_ff], W_down_s[d_ff][d] right after its W_down.
 * A blob of any other size returns TTT_ERR_ARG.
 */
TTT_API int ttt_load_weights(ttt_ctx* ctx, const float* host_blob, size_t n_floats);

/*
 * One inner-loop step for every sequence.
 *   tokens      host int32 [n_seqs][n], the next n tokens of each sequence (1 <= n <= b)
 *   next_tokens host int32 [n_seqs], the token after the chunk (target of its last
 *               position), -1 at the end of the sequence
 *   chunk_loss  host float [n_seqs], out: mean cross-entropy over the chunk's
 *               valid targets, computed with the fast weights before this step
 * The fast weights are then updated and the position advances by n.  Blocks
 * until the losses are on the host.
 */
TTT_API int ttt_prefill_chunk(ttt_ctx* ctx, const int32_t* tokens, int32_t n, const int32_t* next_tokens,
                      float* chunk_loss);

/*
 * Same step with DEVICE buffers, enqueued on the context stream without any
 * synchronisation: d_tokens int32 [n_seqs][n], d_next int32 [n_seqs],
 * d_loss float [n_seqs] (written when the work completes).  Token ids are
 * checked on the device; a bad id is reported by the next ttt_sync.
 */
TTT_API int ttt_prefill_chunk_dev(ttt_ctx* ctx, const int32_t* d_tokens, int32_t n, const int32_t* d_next,
                          float* d_loss);

/*
 * Whole sequences with DEVICE buffers: d_tokens int32 [n_seqs][T], d_losses
 * float [n_seqs][ceil(T/b)].  Equivalent to ceil(T/b) calls of
 * ttt_prefill_chunk_dev in order (targets run across chunk boundaries; the
 * last position has none).  Asynchronous like ttt_prefill_chunk_dev.
 */
TTT_API int ttt_prefill_sequence_dev(ttt_ctx* ctx, const int32_t* d_tokens, int32_t T, float* d_losses);

/*
 * Whole sequences with HOST buffers: tokens int32 [n_seqs][T] (checked on the
 * host: ids in [0, vocab)), losses float [n_seqs][ceil(T/b)], out.  The
 * tokens go to the device in one copy, the sequence runs as in
 * ttt_prefill_sequence_dev, and the losses come back in one copy; blocks
 * until they are on the host.  The context keeps a device staging buffer for
 * the tokens and losses, grown (one cudaMalloc) when a longer T comes in.
 */
TTT_API int ttt_prefill_sequence(ttt_ctx* ctx, const int32_t* tokens, int32_t T, float* losses);

/*
 * Decode-phase TTT with DEVICE buffers (pages: "TTT-E2E技术：突破大语言模型上下文限制的新范式",
 * §2.2 "批量更新与稳定性控制": one update per chunk of input tokens while prefilling and
 * one per chunk of generated tokens while generating; "把 Transformer 做成“终身学习者”",
 * §4.2: the inner loop is reused at inference).  For every sequence:
 *   1. the prompt (d_prompt int32 [n_seqs][T]) goes through the chunked inner loop
 *      as in ttt_prefill_sequence_dev (its last position has no target);
 *      chunk losses -> d_prefill_losses float [n_seqs][ceil(T/b)];
 *   2. the token at position t is picked from the logits of position t - 1, as the
 *      forward of t - 1's chunk computes them, before that chunk's update; the first
 *      one comes from the prompt's last position.  sample = 0: the first index of
 *      the largest logit; sample = 1: inverse CDF of softmax(z / temp) at the caller's
 *      uniform u[i] (d_u float [n_seqs][n_new + 1], in [0, 1)) -- the first index
 *      whose running sum of exp(z/temp - max) exceeds u[i] times the total;
 *   3. generated tokens form chunks of b from the first generated position; each
 *      complete chunk takes one inner-loop step (forward, mean next-token loss whose
 *      last target is the token picked after the chunk, suffix backward, SGD, cache
 *      commit) -> d_gen_losses float [n_seqs][n_new / b] (may be NULL if n_new < b);
 *      an incomplete last chunk takes no step.
 * d_out int32 [n_seqs][n_new + 1]: the n_new generated ids, then the id picked after
 * them.  d_logits (optional) float [n_seqs][n_new + 1][V]: the logits row behind each
 * pick.  Every generated token is one forward over one row per block (bf16 or split
 * products as in prefill); ids never leave the device.  Asynchronous like the other
 * _dev calls; sequences continue from their current position and fast weights.
 */
TTT_API int ttt_decode_dev(ttt_ctx* ctx, const int32_t* d_prompt, int32_t T, int32_t n_new, int32_t sample,
                           float temp, const float* d_u, int32_t* d_out, float* d_prefill_losses,
                           float* d_gen_losses, float* d_logits);

/* Wait for the context stream and report a device-side error (TTT_ERR_DEVICE). */
TTT_API int ttt_sync(ttt_ctx* ctx);

/*
 * Copy the current fast weights of trainable block `suffix_layer` (0 = block
 * L-S, ..., S-1 = block L-1) of sequence `seq` to host memory:
 * w_up float [d][d_ff], w_down float [d_ff][d] (either may be NULL).
 */
TTT_API int ttt_get_fast_weights(ttt_ctx* ctx, int32_t seq, int32_t suffix_layer, float* w_up, float* w_down);

/*
 * Copy the key/value window cache of block `layer` of sequence `seq` to host
 * memory (for checks and state export): k_out, v_out float [window][d_model]
 * (post-RoPE keys; the value of each bf16 operand, plus its remainder in the
 * fp32 mode); pos_out int64 [window], the absolute position whose keys/values
 * slot i holds (the latest p < position with p mod window == i), -1 if none.
 * Any output may be NULL.  Synchronises the context stream.
 */
TTT_API int ttt_get_window(ttt_ctx* ctx, int32_t seq, int32_t layer, float* k_out, float* v_out, int64_t* pos_out);

/*
 * Resumable state of one sequence (pages: "TTT-E2E技术：突破大语言模型上下文限制的新范式",
 * §5.1, the adapted "personal parameters" kept per user; "把 Transformer 做成“终身学习者”",
 * §4.2, the window cache the next chunk reads): its position, its fp32 fast
 * weights and its key/value window cache, as one host byte buffer.
 *   ttt_state_bytes   size of that buffer for this context's shape (-1 for NULL)
 *   ttt_export_state  synchronises the context stream, then copies sequence
 *                     `seq`'s state into host_buf (exactly ttt_state_bytes bytes)
 *   ttt_import_state  replaces sequence `seq`'s state by an exported one; the
 *                     context must be loaded and of the same shape (layers,
 *                     trainable blocks, widths, window, compute mode, dual-MLP),
 *                     else TTT_ERR_ARG; the fast weights' bf16 shadows are derived
 *                     again on the device.  Synchronises.
 * Layout: a 48-byte header ("TTTSTAT1", L, S, d, d_ff, window, fp32 mode,
 * dual-MLP, pad, int64 position), W_up fp32 [S][d][d_ff], W_down fp32
 * [S][d_ff][d], then the cache keys and values bf16 [L][window][d] (then
 * their bf16 remainders in the fp32 mode), slot = position mod window.
 * Exporting after chunk i and importing into a fresh context continues the
 * sequence from chunk i + 1 with the same results.
 */
TTT_API int64_t ttt_state_bytes(const ttt_ctx* ctx);
TTT_API int ttt_export_state(ttt_ctx* ctx, int32_t seq, void* host_buf, size_t bytes);
TTT_API int ttt_import_state(ttt_ctx* ctx, int32_t seq, const void* host_buf, size_t bytes);

/*
 * Restart every sequence from the loaded weights without re-uploading them:
 * position 0, empty window cache, fast weights = the loaded W_up / W_down.
 * Enqueued on the context stream.
 */
TTT_API int ttt_reset(ttt_ctx* ctx);

/*
 * on = 1 (the default): within a sequence, the frozen-block pass of the next
 * group of chunks runs on a second stream of the context beside the current
 * group's trainable steps, and the fast-weight gradient products with their SGD
 * step run on a third stream beside the rest of each chunk's backward; with
 * several sequences, up to 4 of them run side by side, each on its own lane
 * (working buffers and streams), their launches enqueued chunk by chunk in turn.
 * on = 0: every kernel runs on the context stream in issue order, one sequence
 * after another (per-kernel timings then measure each kernel alone).  Results
 * are the same either way, up to the summation order of K-sliced products.
 * Synchronises the context stream; returns TTT_ERR_ARG for another value.
 */
TTT_API int ttt_set_concurrency(ttt_ctx* ctx, int32_t on);

/* Kernels launched by this context since it was created (monotonic counter). */
TTT_API int64_t ttt_launch_count(const ttt_ctx* ctx);

/*
 * Per-kernel-class timing.  ttt_profile(ctx, mask) synchronises, clears the
 * accumulators and starts bracketing with CUDA events (on the context stream)
 * every launch whose class bit is set in `mask` (bit i = class i, named by
 * ttt_profile_class_name(i); -1 = every class; 0 = off).  ttt_profile_read
 * synchronises, folds the recorded launches into the accumulators and writes
 * up to max_out entries (classes with at least one launch); *n_out = number
 * of such classes.  alg_flops counts the multiply-adds the method needs (x2),
 * exec_flops what the kernels execute (masked attention tiles, logit
 * recompute, split-mode triple products), bytes the algorithmic HBM traffic
 * of memory-bound classes.
 */
typedef struct {
  char name[32];
  int64_t launches;
  double ms;
  double alg_flops;
  double exec_flops;
  double bytes;
} ttt_kernel_stat;
TTT_API int ttt_profile(ttt_ctx* ctx, int64_t class_mask);
/*
 * Bracket only one launch in `every` (>= 1; 1, the default, brackets all) of
 * each profiled class, counted in issue order from the next ttt_profile call.
 * An event between two launches ends the overlap of programmatic dependent
 * launch there, so sampling keeps the timed work closer to an unprofiled run.
 * Returns TTT_ERR_ARG for every < 1.
 */
TTT_API int ttt_profile_sample(ttt_ctx* ctx, int32_t every);
/* Name of kernel class `cls` (0-based), NULL past the last class. */
TTT_API const char* ttt_profile_class_name(int cls);
TTT_API int ttt_profile_read(ttt_ctx* ctx, ttt_kernel_stat* out, int max_out, int* n_out);

/* Current absolute position (tokens consumed) of every sequence. */
TTT_API int64_t ttt_position(const ttt_ctx* ctx);

TTT_API void ttt_destroy(ttt_ctx* ctx);

/* Text of the last error on this context ("" if none); valid until the next call. */
TTT_API const char* ttt_last_error(const ttt_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* TTT_H */

/*
 * ns.h -- C ABI of a single-GPU (GB300, sm_103a) continuous-batching transformer decode step
 * over a paged KV cache.
 *
 * What the step computes (per request row, independently): embedding gather; per layer a
 * pre-norm decoder block -- RMSNorm, QKV projection, RoPE, paged KV-cache write, paged
 * grouped-query decode attention, O projection + residual, RMSNorm, SwiGLU FFN + residual;
 * then a final RMSNorm and the LM head to fp32 logits.  Sources, by page and section:
 *   - "GPU waiting, not working" (nanoserve notes), the table under "What I changed because
 *     of it": RoPE cos/sin once per step, fused RMSNorm, grouped-query attention without the
 *     expanded K/V copy, one pinned host-to-device copy of step metadata, token-to-slot
 *     mapping, a fused paged-attention kernel; "Where this leaves nanoserve": capture the
 *     decode step as CUDA graphs once and replay them.
 *   - "NanoFlow: LLM Serving Is Compute Bound, and Your GPU Is Half Idle": "Four resource
 *     classes" (dense KQV/O/Up/Gate/Down, memory-bound decode attention), "Nano-batching:
 *     manufacturing independence" (split the dense batch, co-run nano-ops of different
 *     resource classes), "The part that is harder than it looks" (thread-block budgets per
 *     nano-op), closing paragraph (CUDA events order nano-ops).
 *   - "Speeding up model cold start", "Bounding the CUDA graph capture": capture graphs only
 *     for the batch sizes actually used.
 *
 * Conventions for every call:
 *   - Every call returns ns_status; nothing aborts the process.  Host-side validation fails
 *     before anything is launched or changed.  CUDA runtime failures map to NS_ERR_CUDA and
 *     ns_last_error_message() gives the text.
 *   - "device" pointers are CUDA device memory of the current device; "host" pointers are
 *     ordinary (pageable or pinned) host memory.  The library never frees caller memory.
 *   - Work is enqueued on the caller's `stream` (a cudaStream_t; NULL = legacy default) and
 *     the call returns after enqueueing.
 *   - A handle is not thread safe: one thread at a time per handle.
 *   - Kernels check indices they read from metadata (block ids, slots, lengths).  A failed
 *     check, or a wait inside a kernel that runs past its time limit, skips the access and
 *     records a code that ns_get_device_error() returns; kernels never trap.
 */
#ifndef NS_DECODE_STEP_H
#define NS_DECODE_STEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ns_stream_t; /* same type as cudaStream_t */

typedef enum {
  NS_OK = 0,
  NS_ERR_INVALID_ARG = 1,     /* argument out of range or inconsistent; nothing launched */
  NS_ERR_OUT_OF_MEMORY = 2,   /* device or pinned allocation failed */
  NS_ERR_CUDA = 3,            /* a CUDA runtime / driver call failed */
  NS_ERR_UNSUPPORTED = 4,     /* shape or dtype this library does not implement */
  NS_ERR_NOT_INITIALIZED = 5, /* e.g. ns_decode_step before ns_kv_alloc */
  NS_ERR_DEVICE_CHECK = 6,    /* a kernel recorded a failed bounds check or a timed-out wait */
  NS_ERR_OUT_OF_BLOCKS = 7    /* the KV block pool has too few free blocks */
} ns_status;

typedef enum { NS_F16 = 0, NS_BF16 = 1 } ns_dtype;

/* Device error codes recorded by kernels (ns_get_device_error). */
enum {
  NS_DEV_OK = 0,
  NS_DEV_BAD_BLOCK = 1,    /* block id outside the pool */
  NS_DEV_BAD_SLOT = 2,     /* slot outside the pool */
  NS_DEV_BAD_LENGTH = 3,   /* seq_len outside [1, max_blocks_per_seq * block_size] */
  NS_DEV_WAIT_TIMEOUT = 4, /* an mbarrier wait exceeded its time limit (the kernel returned) */
  NS_DEV_BAD_TOKEN = 5     /* token id outside the vocabulary */
};

typedef struct ns_ctx* ns_handle;

/* Model configuration.  Dims: hidden H, n_layers L, n_q_heads Hq, n_kv_heads Hkv (Hq % Hkv
 * == 0, G = Hq / Hkv <= 8), head_dim d in {64, 128}, ffn F, vocab V.  This library requires
 * H, Hq*d, Hkv*d, 2F, V multiples of 128 and H, Hq*d, F multiples of 64.
 * rope_theta: RoPE base; pairs (i, i + d/2), inverse frequency theta^(-2i/d).
 * rms_eps: RMSNorm epsilon, y = x / sqrt(mean(x^2) + eps) * gamma.
 * max_batch: largest batch ns_decode_step accepts (rows; <= 4096).
 * max_blocks_per_seq: width of the block table rows passed to ns_decode_step (<= 4096).
 * use_graphs: 1 = capture the step as a CUDA graph per batch size on first use and replay
 * it; 0 = launch the kernels eagerly every step (a debugging path). */
typedef struct {
  int hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  float rms_eps;
  double rope_theta;
  int dtype; /* ns_dtype: storage type of weights, activations and the KV cache */
  int tie_embeddings;
  int max_batch, max_blocks_per_seq, use_graphs;
} ns_model_cfg;

/* One layer's weights (host or device pointers, storage dtype).  Linear weights are row-major
 * [out_features][in_features] (y = x W^T): wq [Hq*d][H], wk/wv [Hkv*d][H], wo [H][Hq*d],
 * w_gate/w_up [F][H], w_down [H][F]; attn_norm/ffn_norm are the RMSNorm gains [H]. */
typedef struct {
  const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
} ns_layer_weights;

/* embed [V][H]; final_norm [H]; lm_head [V][H] or NULL when tie_embeddings (head = embed). */
typedef struct {
  const void *embed, *final_norm, *lm_head;
  const ns_layer_weights* layers; /* [n_layers] */
} ns_weights;

/* Create a handle on the current device.  Copies and re-lays-out the weights into
 * library-owned device memory (QKV concatenated, gate/up interleaved in 64-row groups), so
 * the caller may free its copies on return.  Creates the streams, events and TMA descriptors
 * the step uses.  Errors: INVALID_ARG (bad dims/pointers), UNSUPPORTED (shape this library
 * does not implement), OUT_OF_MEMORY, CUDA. */
ns_status ns_create(const ns_model_cfg* cfg, const ns_weights* w, ns_handle* out);

/* Free everything the handle owns (device memory, graphs, streams).  NULL is ignored. */
void ns_destroy(ns_handle h);

/* Allocate the per-layer paged K and V pools: num_blocks blocks of block_size (16) token
 * slots.  Layout per layer and per K/V: [num_blocks][Hkv][block_size][d], storage dtype, so
 * each (block, kv head) tile is contiguous; one more block follows each pool, reserved for the
 * padding rows of bucketed graphs (ns_set_graph_buckets).  Initialises the host free list 0..num_blocks-1
 * (first-in first-out reuse).  A second call returns INVALID_ARG. */
ns_status ns_kv_alloc(ns_handle h, int num_blocks, int block_size);

/* Device addresses of layer `layer`'s K and V pools (for preloading synthetic context). */
ns_status ns_kv_layer_ptrs(ns_handle h, int layer, void** k_pool, void** v_pool);

/* Host slot mapper ("mapping tokens to cache slots", nanoserve notes).  For each row b in
 * order: p = positions[b]; when p % block_size == 0 a block is popped from the free list into
 * block_tables[b][p / block_size]; slot_mapping[b] = block_tables[b][p/bs] * bs + p % bs.
 * block_tables: host, [batch][max_blocks_per_seq] int32, updated in place.  slot_mapping: host,
 * [batch] int64, written.  Fails with OUT_OF_BLOCKS / INVALID_ARG before changing anything. */
ns_status ns_kv_prepare_step(ns_handle h, int batch, const int32_t* positions,
                             int32_t* block_tables, int64_t* slot_mapping);

/* Host-only block pool (no GPU needed): the free list and slot mapper that a handle's KV cache
 * uses, usable on its own.  Same policy as ns_kv_prepare_step / ns_kv_reserve / ns_kv_release:
 * the free list starts 0..num_blocks-1, blocks are taken from the front and returned to the
 * back, and only blocks handed out can be returned (once).  max_blocks_per_seq is the
 * block-table row width prepare_step writes into. */
typedef struct ns_block_pool* ns_pool;
ns_status ns_pool_create(int num_blocks, int block_size, int max_blocks_per_seq, ns_pool* out);
void ns_pool_destroy(ns_pool p);
ns_status ns_pool_prepare_step(ns_pool p, int batch, const int32_t* positions,
                               int32_t* block_tables, int64_t* slot_mapping);
ns_status ns_pool_reserve(ns_pool p, int n, int32_t* out_ids);
ns_status ns_pool_release(ns_pool p, const int32_t* block_ids, int n);
ns_status ns_pool_free_count(ns_pool p, int* n_free);
ns_status ns_pool_geometry(ns_pool p, int* num_blocks, int* block_size);

/* The pool a handle's KV cache allocates from (after ns_kv_alloc), for the batch former below.
 * Borrowed: it lives as long as the handle; never pass it to ns_pool_destroy. */
ns_status ns_kv_get_pool(ns_handle h, ns_pool* out);

/* Constant-dense-batch former (NanoFlow page, "Runtime details that keep the pipeline fed": the
 * scheduler keeps the batch at the size the overlap schedule was tuned for by taking the
 * unfinished decode requests first and topping up with prefill chunks cut at token
 * granularity; requests that exceed their predicted peak memory go to the host and are
 * reloaded later, never recomputed).  Host only; no GPU needed.  Each step:
 *   ns_sched_next fills the metadata of ns_decode_step for at most dense_tokens rows:
 *   1. while the decode rows of the first dense_tokens running requests need more new blocks
 *      than are free, the last running request is preempted: a save move lists its cached
 *      tokens (positions 0 .. prompt_len + generated - 2) and its blocks, the blocks return to
 *      the pool, and it waits;
 *   2. in a step that preempted nothing, waiting preempted requests resume, first in first out,
 *      while the free blocks (after this step's decode blocks) hold the blocks of their cached
 *      tokens and of their next position: a reload move lists the new blocks, and the request
 *      runs again (last in the running order);
 *   3. one decode row per running request, in running order (prompt completion order, resumed
 *      requests appended), at most dense_tokens; a decode row's token is the request's last
 *      sampled token at position prompt_len + generated - 1;
 *   4. prompts in arrival order, each adding its next min(room, remaining) tokens as
 *      consecutive positions over its own block table, cut to what the free blocks hold; a
 *      prompt starts only when the free blocks cover its predicted peak -- the blocks of its
 *      first prompt_len + min(max_new_tokens, predicted_new_tokens) - 1 positions
 *      (predicted_new_tokens 0: max_new_tokens) -- plus what the requests holding blocks still
 *      need to reach their predicted peaks and what the preempted ones need to resume; the fill
 *      stops at the first prompt that gets no row.
 *   Blocks are reserved as positions cross block boundaries, in row order.  seq_lens =
 *   positions + 1; every chunk row carries its request's whole block table, so a prompt's rows
 *   see one another causally within the step (ns_decode_step).  Arrays are host memory of
 *   dense_tokens rows (block_tables [dense_tokens][max_blocks_per_seq]); row_request[b] is the
 *   request of row b and row_samples[b] = 1 where the row yields a token (decode rows and a
 *   prompt's last row).  *batch may be 0 (nothing to run).
 *   ns_sched_moves lists the step's moves, saves first: the caller performs them in that order
 *   on the step's stream before ns_decode_step (ns_kv_save of kind 0 into its own host store,
 *   ns_kv_reload of kind 1 from it; a reload's blocks may be blocks a save of the same step
 *   released, which stream order makes safe).
 *   A prompt whose last row is formed joins the running order at once (its next decode row
 *   comes in the following step).
 *   ns_sched_commit then takes the step's sampled tokens (sampled[b], read where
 *   row_samples[b] = 1; batch must equal the formed step's, else INVALID_ARG and nothing
 *   changes): a request that samples eos_token or reaches max_new_tokens finishes, its blocks
 *   return to the pool in table order, and its id is written to finished_ids (capacity >=
 *   batch, or NULL).  A second ns_sched_next before the commit returns INVALID_ARG.
 * With predicted_new_tokens 0 every admitted request's peak is reserved, so nothing is ever
 * preempted. */
typedef struct ns_sched_st* ns_sched;
/* pool is borrowed: it must outlive the former, and while the former runs only the former
 * reserves and releases its blocks.  dense_tokens >= 1 (the target rows per step),
 * max_blocks_per_seq >= 1 (the row width of the block tables it writes), eos_token (any
 * value; one no token equals disables eos), predicted_new_tokens >= 0; else INVALID_ARG. */
ns_status ns_sched_create(ns_pool pool, int dense_tokens, int max_blocks_per_seq, int eos_token,
                          int predicted_new_tokens, ns_sched* out);
void ns_sched_destroy(ns_sched s);
/* prompt: host, prompt_len >= 1 non-negative token ids (copied; negative ids are reserved for
 * rows that read a device-sampled token); prompt_len + max_new_tokens at most
 * max_blocks_per_seq * block_size, and its blocks at most the pool's; ids are unique and
 * non-negative. */
ns_status ns_sched_add(ns_sched s, int request_id, const int32_t* prompt, int prompt_len,
                       int max_new_tokens);
ns_status ns_sched_next(ns_sched s, int32_t* token_ids, int32_t* positions, int32_t* block_tables,
                        int32_t* seq_lens, int64_t* slot_mapping, int32_t* row_request,
                        int32_t* row_samples, int* batch);
/* The formed step's moves: *n = their count, the first min(*n, capacity) written (tables:
 * [capacity][max_blocks_per_seq], the request's blocks in table order, zero-padded). */
ns_status ns_sched_moves(ns_sched s, int32_t* kinds, int32_t* request_ids, int32_t* n_tokens,
                         int32_t* tables, int capacity, int* n);
ns_status ns_sched_commit(ns_sched s, const int32_t* sampled, int batch, int32_t* finished_ids,
                          int* n_finished);
/* Tokens generated so far by a request (running, preempted or finished): *n = their count, the
 * first min(*n, capacity) copied to out. */
ns_status ns_sched_tokens(ns_sched s, int request_id, int32_t* out, int capacity, int* n);
/* Requests with prompt tokens left, running, preempted, and finished ones not yet removed. */
ns_status ns_sched_counts(ns_sched s, int* waiting, int* running, int* preempted, int* finished);
/* Forget a finished request (its tokens and id); INVALID_ARG for an unknown or unfinished id, or
 * while a formed row of it is not committed.  A long-running caller removes requests once it has
 * read their tokens. */
ns_status ns_sched_remove(ns_sched s, int request_id);
/* Asynchronous formation (NanoFlow page, "Runtime details that keep the pipeline fed": the batch
 * of iteration i + 1 is formed before iteration i finishes, so an end-of-sequence token is seen
 * one iteration late).  With on != 0, ns_sched_next may be called once while one formed step is
 * not committed yet; ns_sched_commit then commits the oldest.  A decode row whose token is not
 * committed yet gets token id -(row + 1): the token sampled at that row of the previous step,
 * which ns_decode_step reads from the device token source (ns_set_token_source; the previous
 * step's greedy ids).  A request counts its formed rows toward max_new_tokens; one that samples
 * eos_token keeps the row already formed for it in the next step (its token is ignored at that
 * step's commit) and returns its blocks when no formed row of it is uncommitted.  Needs
 * predicted_new_tokens = 0 (every peak reserved, so nothing is ever preempted) and no formed
 * step pending, else INVALID_ARG.  A prompt joins the running order when its last row is formed,
 * in either mode. */
ns_status ns_sched_set_async(ns_sched s, int on);

/* Host validation of one step's metadata, exactly as ns_decode_step performs it before
 * anything is launched: 1 <= batch <= max_batch; token ids in [0, vocab); positions >= 0;
 * seq_lens == positions + 1 <= max_blocks_per_seq * block_size; the first
 * ceil(seq_len / block_size) table entries in [0, num_blocks); slot_mapping[b] ==
 * block_tables[b][p / bs] * bs + p % bs.  Returns NS_OK or NS_ERR_INVALID_ARG. */
ns_status ns_check_step_metadata(int num_blocks, int block_size, int max_blocks_per_seq,
                                 int vocab, int max_batch, int batch, const int32_t* token_ids,
                                 const int32_t* positions, const int32_t* block_tables,
                                 const int32_t* seq_lens, const int64_t* slot_mapping);

/* Reserve n blocks from the free list (host ids written to out_ids[n]); OUT_OF_BLOCKS if short. */
ns_status ns_kv_reserve(ns_handle h, int n, int32_t* out_ids);

/* Return blocks to the back of the free list (a request leaving).  A block has one owner, so
 * every id must be one that was handed out (reserve, prepare_step, the batch former) and not
 * yet returned, and appear once in the call; INVALID_ARG otherwise (an id outside the pool, a
 * free block, a repeated id), with nothing returned. */
ns_status ns_kv_release(ns_handle h, const int32_t* block_ids, int n);

/* Number of free blocks. */
ns_status ns_kv_free_count(ns_handle h, int* n_free);

/* Nano-batching (NanoFlow page, "Nano-batching: manufacturing independence"): split each
 * step's rows into n_split (1..4) consecutive nano-batches of the given sizes (host array;
 * NULL = even split rounded to multiples of 128 where possible).  Nano-batch i runs on stream
 * i % 2; its attention waits on the QKV projection of every earlier nano-batch of the same
 * layer (prefill rows of one chunk may span nano-batches); everything else in a nano-batch
 * depends only on its own rows, so results are bitwise identical to the unsplit step.
 * attn_cta_budget > 0 caps the attention grid (thread blocks) of each nano-op, <= 0 = one
 * wave.  Sizes must sum to the batch of the following ns_decode_step calls. */
ns_status ns_set_nanobatch(ns_handle h, int n_split, const int* sizes, int attn_cta_budget);

/* The other half of the NanoFlow page's per-nano-op thread-block budgets ("The part that is
 * harder than it looks"): in nano-batched steps (n_split > 1), projections that run the
 * persistent GEMM (more than 64 rows of an unsplit weight with two 256-token output tiles per
 * SM) use at most gemm_cta_budget CTAs, one per SM, so the other nano-batch's attention can take
 * the SMs they leave free; 0 = one per SM.  The persistent GEMM computes every output tile the
 * same way on any grid, so results are bitwise unchanged.  gemm_cta_budget < 0 returns
 * INVALID_ARG.  Unsplit steps ignore it. */
ns_status ns_set_gemm_cta_budget(ns_handle h, int gemm_cta_budget);

/* How a step is run ("The chef who calls out every order" and "The maths that matters: when the
 * GPU is left waiting" in the nanoserve notes: at small batch a decode step is a chain of short
 * kernels whose launch and dependency waits cost more than their own weight reads).
 *   mode 0 (the default): one kernel per stage (embedding, per layer QKV, attention, O,
 *     gate/up, down, then the LM head), captured in a graph when the handle uses graphs.
 *   mode 1: steps of at most 32 decode rows, without nano-batches, prefill chunks, KV offload,
 *     trace or per-kernel timing, run as one persistent cooperative kernel with one CTA per SM
 *     (a grid-wide barrier between stages, each CTA streaming its share of every layer's weights
 *     into shared memory ahead of the stages); other steps keep mode 0's kernels.
 * The first switch to mode 1 packs a second copy of every projection weight and of the LM head
 * (the handle's weight bytes again) into per-CTA streams and allocates small step buffers;
 * mode 0 keeps them for a later switch back, ns_destroy frees them.  The two modes sum in
 * different orders, so a row's bits differ between them (both are checked against the oracle);
 * within mode 1 a row's result depends only on its own inputs, as in mode 0.  Graphs are
 * cached per mode.  UNSUPPORTED when head_dim is not 64 or 128, a KV head serves more than 8
 * query heads, ffn is not a multiple of 128 or hidden exceeds 4096; OUT_OF_MEMORY when the packed copy does not
 * fit.  mode outside {0, 1}: INVALID_ARG. */
ns_status ns_set_step_kernel(ns_handle h, int mode);

/* One decode step for `batch` rows.  Host metadata (validated, packed into one pinned buffer
 * and uploaded with a single host-to-device copy on `stream`):
 *   token_ids [batch] int32 in [0, V) (with a device token source set, NULL or entries
 *   -(r + 1) too: see ns_set_token_source); positions [batch] int32 >= 0;
 *   block_tables [batch][max_blocks_per_seq] int32 (entries for blocks 0..ceil(seq_len/bs)-1
 *   must be valid pool ids; the rest are ignored); seq_lens [batch] int32 == positions + 1
 *   (cached tokens including this step's token); slot_mapping [batch] int64, must equal
 *   block_tables[b][p/bs]*bs + p%bs.
 * logits_out: device, [batch][V] fp32, written; NULL stops the step after the last layer
 * (no final norm, no LM head), for callers that only advance the KV cache or time the layers
 * alone.  Writes this step's K/V into the pools; every row's K/V is written before any row
 * attends, so rows of one prompt chunk (consecutive positions over one block table) see each
 * other causally.  Working back from the last row, each maximal run of at least 16 such rows
 * whose tables agree with the run's last row is a prompt chunk attended by one causal
 * prefill-chunk kernel (so a step may end with several chunks, one per prompt); the search
 * stops at the first shorter run, and the rows before it use the decode kernel.
 * With use_graphs the first call for a batch size (or graph bucket) captures a graph (not
 * during a caller's stream capture); later calls replay it.  Returns NOT_INITIALIZED before
 * ns_kv_alloc. */
ns_status ns_decode_step(ns_handle h, int batch, const int32_t* token_ids,
                         const int32_t* positions, const int32_t* block_tables,
                         const int32_t* seq_lens, const int64_t* slot_mapping,
                         float* logits_out, ns_stream_t stream);

/* The prompt chunks ns_decode_step would find in a step (host only, no GPU): the first row of
 * each, in row order.  Working back from the last row, each maximal run of at least 16 rows at
 * consecutive positions whose first ceil(seq_len / block_size) block-table entries equal those
 * of the run's last row is one chunk; the first shorter run ends the search.  Host arrays of
 * `batch` rows (block_tables [batch][max_blocks_per_seq]); seq_lens in [1, max_blocks_per_seq
 * * block_size] and positions >= 0, else INVALID_ARG.  *n = the number of chunks; the first
 * min(*n, capacity) starts are written. */
ns_status ns_find_prompt_chunks(int block_size, int max_blocks_per_seq, int batch,
                                const int32_t* positions, const int32_t* block_tables,
                                const int32_t* seq_lens, int32_t* starts, int capacity, int* n);

/* Graph buckets ("Bounding the CUDA graph capture", model cold-start page: capture graphs for
 * a bounded set of batch sizes and pad).  With n > 0 ascending sizes (each <= max_batch), a
 * graph-replayed step of `batch` rows uses the graph of the smallest size >= batch; the rows
 * up to that size are padding (token 0 at position 0 in a block past the caller's pool, no
 * logits written), so one captured graph serves every batch up to its size.  Batches above the
 * largest size, eager steps and nano-batched steps use their exact size.  n = 0 clears. */
ns_status ns_set_graph_buckets(ns_handle h, int n, const int* sizes);

/* Whether steps with prompt chunks (see ns_decode_step) replay graphs (capture != 0, the
 * default) or launch eagerly (0).  A batch former's mixed steps rarely repeat a chunk layout, and
 * every new layout is a new capture; with 0 only decode-only steps use (and capture) graphs. */
ns_status ns_set_graph_chunks(ns_handle h, int capture);

/* Token ids from device memory (NanoFlow page, "Runtime details that keep the pipeline fed":
 * the next iteration's batch is formed before the current one finishes, so an end-of-sequence
 * token is seen one iteration late and no synchronisation sits on the critical path).  When
 * device_token_ids is non-NULL (int32, device memory of at least max_batch entries, owned by
 * the caller), every later ns_decode_step may take tokens from it: with token_ids NULL, row b
 * reads device_token_ids[b]; with token_ids given, an entry -(r + 1) (1 <= r + 1 <= max_batch)
 * makes row b read device_token_ids[r] and an entry in [0, V) is used as is (the form the batch
 * former's asynchronous mode writes, ns_sched_set_async).  A device token outside [0, V) sets
 * NS_DEV_BAD_TOKEN and the row uses token 0.  Writes to the buffer must be ordered before the
 * step on its stream (for example ns_greedy_argmax of the previous step's logits on the same
 * stream).  NULL restores host token ids only (negative ids are then INVALID_ARG).  A graph is
 * captured per source pointer. */
ns_status ns_set_token_source(ns_handle h, const int32_t* device_token_ids);

/* KV offload (NanoFlow page, "Runtime details that keep the pipeline fed": K/V go to the host
 * right after the QKV projection produces them, while they are still contiguous, and the copy
 * overlaps the FFN).  With host_dst non-NULL, every later ns_decode_step also writes the K (after
 * RoPE) and V that it stores for row b of layer l into row (l, b) of host_dst, laid out
 * [n_layers][max_batch][2][n_kv_heads * head_dim] in the model dtype (K first, then V; the same
 * bits as the cache).  The QKV epilogue stages the rows in a device buffer of that layout and a
 * copy stream moves each layer's rows to host_dst as soon as that layer's QKV finishes, while its
 * attention and FFN run; the step's work on its stream completes only after every copy has.
 * Rows batch .. max_batch-1 are unspecified (graph padding rows land there).  host_dst must be
 * pinned host memory (cudaMallocHost or cudaHostRegister, else NS_ERR_INVALID_ARG) of at least
 * bytes = n_layers * max_batch * 2 * n_kv_heads * head_dim * 2 bytes, owned by the caller; each
 * step overwrites it, so copy a step's rows out before the next step's work starts.  A graph is
 * captured per destination.  NULL stops the mirroring. */
ns_status ns_set_kv_offload(ns_handle h, void* host_dst, size_t bytes);

/* KV reload (same page: reloaded K/V land in one contiguous device buffer and only then are
 * scattered into the fragmented pages, instead of scattering across the host link).
 * host_src holds the K/V of n_tokens tokens of one request at positions first_pos ..
 * first_pos + n_tokens - 1, laid out [n_layers][n_tokens][2][n_kv_heads * head_dim] in the model
 * dtype (the ns_set_kv_offload row layout, one row per token).  They are copied to a contiguous
 * device buffer held by the handle, then scattered to slot block_table[p / bs] * bs + p % bs of
 * every layer's pools, bs the block_size given to ns_kv_alloc (block_table: host int32 of
 * n_table >= (first_pos + n_tokens - 1) / bs + 1 ids in [0, num_blocks), else
 * NS_ERR_INVALID_ARG).  Asynchronous on `stream`; host_src must stay
 * valid until the copy has run when it is pinned (pageable memory is copied before the call
 * returns).  Calls on one handle share the transfer buffer: order them on one stream, and
 * before any step that reads the blocks.  The buffer grows to the largest request seen (the
 * growth synchronises the device).  Returns NOT_INITIALIZED before ns_kv_alloc. */
ns_status ns_kv_reload(ns_handle h, const void* host_src, int n_tokens, int first_pos,
                       const int32_t* block_table, int n_table, ns_stream_t stream);

/* The inverse of ns_kv_reload, for a request whose K/V were not mirrored: the tokens' K/V are
 * gathered from the pages into the contiguous device buffer, then copied to host_dst in the same
 * [n_layers][n_tokens][2][n_kv_heads * head_dim] layout.  Same arguments, ordering and errors. */
ns_status ns_kv_save(ns_handle h, void* host_dst, int n_tokens, int first_pos,
                     const int32_t* block_table, int n_table, ns_stream_t stream);

/* Paged grouped-query decode attention alone (nanoserve notes: the fused paged-attention
 * kernel; grouped-query attention without the expanded K/V copy).  All pointers device:
 *   q [batch][n_q_heads][head_dim]; k_pool, v_pool [num_blocks][n_kv_heads][block_size]
 *   [head_dim]; block_tables [batch][max_blocks_per_seq] int32; seq_lens [batch] int32 in
 *   [1, max_blocks_per_seq*block_size]; out [batch][n_q_heads][head_dim] (same dtype as q).
 * For q head h the kv head is h / (n_q_heads / n_kv_heads); o = softmax(q.K^T * scale) V over
 * tokens t < seq_len.  The split depends only on seq_len, so results do not depend on the
 * batch.  num_blocks * n_kv_heads * block_size must be below 2^31 and max_blocks_per_seq *
 * block_size at most 65536.
 * Rows split into superchunks of at most 1024 tokens (ceil(ceil(L / 16) / 64) of them), merged
 * by log-sum-exp.  Scratch (partials and counters) is allocated by the library on first use per
 * device and kept until exit.  Slots past seq_len in a row's last block are never used, even
 * if they hold non-finite values.  num_blocks bounds the block ids the kernel accepts.  Supports head_dim
 * 64/128, G <= 8 (G in 1,2,4,7,8), block_size 16.  Not to be called during stream capture
 * the first time on a device (it may allocate). */
ns_status ns_attn_decode(const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, const int32_t* seq_lens, void* out,
                         int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                         int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                         ns_stream_t stream);

/* ns_attn_decode on at most cta_budget CTAs (0: no cap): the thread-block cap that the NanoFlow
 * page ("The part that is harder than it looks") sweeps from 8 to 128 when it profiles a
 * memory-bound op co-running with a GEMM.  The CTAs loop over the work, so any cap >= 1
 * computes the same result bitwise.  cta_budget < 0 returns INVALID_ARG. */
ns_status ns_attn_decode_capped(const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, const int32_t* seq_lens, void* out,
                                int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq, int num_blocks,
                                float scale, int dtype, int cta_budget, ns_stream_t stream);

/* ns_attn_decode without any device allocation, for callers that cannot allocate: code
 * running inside an allocator or memory-pool callback, a plugin whose host process owns every
 * device allocation, or a process that must keep its device footprint fixed after start-up.
 * The source pages have no counterpart of this call; it exists for such callers only.
 * Same arguments and result as ns_attn_decode, plus dev_err: an optional device int (NULL = none)
 * where a failed bounds check inside the kernel is recorded.  The split-K scratch (partials and
 * counters) lives in a fixed buffer inside the library image: 32 MiB of partials and 65,536
 * counters, held by every GPU that loads the library until the process exits.  Requests needing
 * more -- batch * n_kv_heads slots of ceil(max_blocks_per_seq / 64) *
 * (n_q_heads / n_kv_heads) * (head_dim + 2) floats each (rounded up to 16 bytes), or
 * batch * n_kv_heads + 1 counters -- return
 * NS_ERR_INVALID_ARG with a message saying so.  The first call on a device looks up the
 * buffer's device address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  The address is kept per device together with the id of the
 * context it belongs to; after a device reset (a new primary context, the library image loaded
 * again) the next call looks it up again, so it too should come before any capture.  All calls
 * on a device share the buffer and each call leaves its contents behind (the counters are
 * cleared on the call's stream before its kernel): calls whose kernels overlap on the GPU
 * race; order them on one stream. */
ns_status ns_attn_decode_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_tables, const int32_t* seq_lens, void* out,
                                 int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                 int block_size, int max_blocks_per_seq, int num_blocks,
                                 float scale, int dtype, int* dev_err, ns_stream_t stream);

/* Dense projection through the tcgen05 GEMM used by the step (NanoFlow page: the dense
 * class KQV/O/Up/Gate/Down): y[m][n] = sum_k x[m][k] * w[n][k], fp32 out.  w [n][k], x [m][k]
 * device, storage dtype; y device fp32 [m][n].  n % 128 == 0, k % 64 == 0, 1 <= m <= 4096.
 * Uses library-allocated split-K scratch (allocated on first use per device). */
ns_status ns_linear(const void* w, const void* x, float* y, int m, int n, int k, int dtype,
                    ns_stream_t stream);

/* Greedy next token per row: index of the largest logit, ties to the lowest index.
 * logits device [batch][vocab] fp32; out_ids device [batch] int32. */
ns_status ns_greedy_argmax(const float* logits, int batch, int vocab, int32_t* out_ids,
                           ns_stream_t stream);

/* Read and clear the device error word of the handle (NULL handle = the word used by the
 * handle-free calls on the current device).  Synchronises the device.  After
 * NS_DEV_WAIT_TIMEOUT it also clears the attention kernel's counters (split-K arrivals and the
 * unit queue's tickets) of the handle or of the handle-free calls, which a kernel that gave up
 * a wait may have left set; the allocation-free call clears its own before every launch. */
ns_status ns_get_device_error(ns_handle h, int* code);

/* Step statistics: kernels launched per step and per graph, graph count, last capture ms. */
typedef struct {
  int kernels_per_step;     /* kernel launches in one step (eager) / kernel nodes (graph) */
  int graphs_cached;        /* captured batch sizes */
  double last_capture_ms;   /* host time of the last capture + instantiate */
  long long steps;          /* ns_decode_step calls that succeeded */
} ns_step_info;
ns_status ns_get_step_info(ns_handle h, ns_step_info* out);

/* Capture report (model cold-start page, "Bounding the CUDA graph capture": capture costs
 * start-up time, so capture only the batch sizes the workload uses, and measure it).  One
 * entry per captured graph. */
typedef struct {
  int batch;            /* graph batch (bucket) size */
  int n_split;          /* nano-batches */
  int attn_cta_budget;  /* 0: none */
  int with_lm;          /* the graph ends with the LM head */
  int chunk_rows;       /* rows of the trailing prefill chunk (0: decode only) */
  int kv_offload;       /* the graph mirrors K/V to the host */
  int kernels;          /* kernel nodes */
  double capture_ms;    /* host time of capture + instantiate */
  int gemm_cta_budget;  /* 0: none (ns_set_gemm_cta_budget) */
  int attn_queue;       /* decode attention hands out its units from a queue, longest rows first
                           (chosen per step: at least 6 units per CTA) */
} ns_graph_info;
/* *n = the number of graphs; the first min(*n, capacity) entries are written, in key order. */
ns_status ns_get_graph_report(ns_handle h, ns_graph_info* out, int capacity, int* n);

/* Capture the decode-only graphs of these batch sizes now (start-up), with or without the LM
 * head, under the current nano-batch, token-source and offload settings, so that no step pays
 * a capture later (where the rows could hold enough attention units for the unit queue, both
 * attention variants are captured).  Sizes in [1, max_batch]; with nano-batches only their total.  Captures are
 * not replayed (no device work is run).  INVALID_ARG when the handle does not use graphs,
 * NOT_INITIALIZED before ns_kv_alloc. */
ns_status ns_capture_graphs(ns_handle h, int n, const int* batch_sizes, int with_lm);

/* Per-kernel timing of eager steps (for roofline accounting).  While on, ns_decode_step
 * launches the kernels eagerly (graphs are bypassed) with a CUDA event pair around each launch
 * on the stream the kernel runs on.  Kinds: 0 embedding + RoPE table, 1 QKV projection,
 * 2 attention (decode rows and prompt-chunk kernels), 3 O projection, 4 gate/up projection,
 * 5 down projection, 6 LM head; entry 7 is reserved and stays 0.
 * ns_get_kernel_timing synchronises, returns launches and summed milliseconds per kind since
 * the last read, and clears them. */
#define NS_KERNEL_KINDS 8
typedef struct {
  int launches[NS_KERNEL_KINDS];
  double total_ms[NS_KERNEL_KINDS];
} ns_kernel_timing;
ns_status ns_set_kernel_timing(ns_handle h, int on);
ns_status ns_get_kernel_timing(ns_handle h, ns_kernel_timing* out);

/* Per-tensor view inside the step, for parity checks layer by layer (the nanoserve notes'
 * change table fuses RMSNorm, RoPE and grouped-query attention inside each layer, so the
 * layer's intermediate tensors are where a fused kernel's error would first show).  While a
 * trace is set, ns_decode_step launches eagerly (graphs are bypassed) and, for layer `layer`,
 * copies on the step's streams right after the kernel that produces each tensor:
 *   q          [batch][n_q_heads * head_dim] storage dtype: q after the projection and RoPE;
 *   attn       [batch][n_q_heads * head_dim] storage dtype: the attention output o;
 *   resid_mid  [batch][hidden] fp32: the residual after the attention block, x + o Wo^T;
 *   resid_out  [batch][hidden] fp32: the residual after the layer (after the FFN).
 * (k and v are the cache slots the step writes: read them from ns_kv_layer_ptrs.)  Every
 * pointer is a caller-owned device buffer of at least that size, or NULL to skip that tensor.
 * layer < 0 or bufs == NULL turns the trace off; layer >= n_layers returns INVALID_ARG. */
typedef struct {
  void* q;
  void* attn;
  float* resid_mid;
  float* resid_out;
} ns_trace_bufs;
ns_status ns_set_trace(ns_handle h, int layer, const ns_trace_bufs* bufs);

/* Human-readable name of a status; thread-local text of the last failure. */
const char* ns_status_str(ns_status s);
const char* ns_last_error_message(void);

#ifdef __cplusplus
}
#endif
#endif /* NS_DECODE_STEP_H */

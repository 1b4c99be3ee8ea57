// Host runtime behind the C ABI in ns.h: weight re-layout, KV pools and the block allocator,
// the single packed metadata upload per step, the per-batch-size CUDA-graph cache, and the
// two-stream nano-batch schedule.
//
// Sources, by page and section:
//  * "GPU waiting, not working" (nanoserve notes), change table: one pinned host-to-device copy
//    of the step metadata instead of six small ones; mapping tokens to cache slots; RoPE once
//    per step; "Where this leaves nanoserve": capture the decode step once as CUDA graphs and
//    replay them.
//  * "Speeding up model cold start", "Bounding the CUDA graph capture": capture only the batch
//    sizes actually used (graphs are captured lazily, per batch size on first use).
//  * "NanoFlow ...", "Nano-batching: manufacturing independence": split the dense batch into
//    nano-batches whose nano-ops co-run; "The part that is harder than it looks": thread-block
//    budgets per nano-op; closing paragraph: CUDA events order the nano-ops.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <deque>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "ns.h"
#include "ns_host.h"

using namespace ns;

namespace {

thread_local std::string g_msg;

ns_status fail(ns_status s, const std::string& m) {
  g_msg = m;
  return s;
}

#define NS_CUDA(expr)                                                                       \
  do {                                                                                      \
    cudaError_t e_ = (expr);                                                                \
    if (e_ != cudaSuccess)                                                                  \
      return fail(e_ == cudaErrorMemoryAllocation ? NS_ERR_OUT_OF_MEMORY : NS_ERR_CUDA,     \
                  std::string(#expr) + ": " + cudaGetErrorString(e_));                     \
  } while (0)

#define NS_TRY(expr)                 \
  do {                               \
    ns_status s_ = (expr);           \
    if (s_ != NS_OK) return s_;      \
  } while (0)

// ------------------------------------------------------------------------------ TMA maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major [rows][cols] 16-bit matrix; box = 64 columns (128 B, one swizzle row) x box_rows.
ns_status make_tmap(CUtensorMap* m, const void* base, int dtype, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(NS_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dtype == NS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NS_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string(r));
  return NS_OK;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Token tile for m rows: balanced tiles of at most 256, multiple of 16.  From 129 to 256 rows a
// CTA with a short k-range (at most 32 k-blocks) takes tiles of at most 128 instead: twice the
// CTAs hide the pipeline's fill and the epilogue better than the wider tile's operand reuse
// pays for (measured on 4096-wide projections at 256 rows: 22 k-blocks 46 -> 31 us, 16 k-blocks
// 31 -> 27 us; with 56 or 64 k-blocks the 256-wide tile stays faster).  The tile never changes
// a result.
int pick_bn_capped(int m, int cap) {
  const int tiles = (m + cap - 1) / cap;
  int bn = round_up((m + tiles - 1) / tiles, 16);
  return std::max(16, std::min(cap, bn));
}

// Above 256 rows a launch without split-K also compares the two widths by their waves of two
// CTAs per SM, charging each CTA 64 + BN token-columns of work (a fixed cost plus its tile),
// and takes the 128-token tile when that is at least 10 % less (the 4096 x 28672 gate/up
// projection at 512 rows: 1.47 -> 2.95 waves, 160 -> 143 us).
int pick_bn(int m, int kb_per_split, int splits, int n_tiles, int sms) {
  if (m > 128 && m <= 256 && kb_per_split <= 32) return pick_bn_capped(m, 128);
  const int wide = pick_bn_capped(m, kMaxBN);
  if (m <= 256 || splits != 1) return wide;
  const int narrow = pick_bn_capped(m, 128);
  const long long slots = 2LL * sms;
  auto cost = [&](int bn) {
    const long long ctas = static_cast<long long>((m + bn - 1) / bn) * n_tiles;
    return ((ctas + slots - 1) / slots) * (64 + bn);
  };
  return cost(narrow) * 10 <= cost(wide) * 9 ? narrow : wide;
}

// Token tile of the persistent GEMM: the widest balanced tile (up to 256 tokens), so each
// weight tile and each activation tile crosses from L2 to the SMs as few times as possible
// (measured on the LLaMA-3-8B projections at 256 rows and the 70B-shaped ones at 1024 and
// 2048: 256-token tiles beat 128-token ones in every case, by up to 1.9x).
int pick_bn_persistent(int m) { return pick_bn_capped(m, kMaxBN); }

// The persistent kernel takes a launch of more than 64 rows of an unsplit weight when it has at
// least two 256-token output tiles per SM, and any launch of an unsplit weight with four or more
// tiles per SM (a vocabulary-wide head).  A split weight stays on the cluster kernel, whose
// distributed-shared-memory reduction is cheaper than a reduction through global memory
// (measured: the LLaMA-3-8B split-K projections at 256 rows 27-48 us against 50-68 us).  A
// short launch stays there too: the persistent kernel's CTA fills an SM, so under programmatic
// dependent launch it cannot start streaming its weights beside the previous kernel's CTAs
// (measured: the 8B gate/up projection at 256 rows 75 us in the step on clusters against 98
// persistent, though 87 against 83 alone).  Both kernels give a row the same bits.
bool use_persistent(int m, int splits, int n_tiles, int sms) {
  if (splits != 1) return false;
  const long long tiles = static_cast<long long>((m + kMaxBN - 1) / kMaxBN) * n_tiles;
  // a very long launch (a vocabulary-wide head: four or more tiles per SM) streams its weights
  // through the persistent kernel's deep ring at any row count
  return tiles >= 4LL * sms || (m >= kPersistentMinRows && tiles >= 2LL * sms);
}

// Split-K from the weight's shape (never the batch; see also choose_splits_for_handle): about
// one CTA per SM, so every
// cluster of a launch is resident at once; at least two k-blocks per split; at most one
// portable cluster (8 CTAs) per output tile.
void choose_splits(int N, int K, int sms, int* splits, int* kb_per) {
  const int tiles = N / kGemmTileN, nkb = K / kGemmTileK;
  int s = std::max(1, sms / std::max(1, tiles));
  s = std::min(s, std::max(1, nkb / 2));
  s = std::min(s, kMaxSplits);
  *kb_per = (nkb + s - 1) / s;
  *splits = (nkb + *kb_per - 1) / *kb_per;
}

int device_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// fp16 / bf16 bit patterns to float (IEEE 754 binary16 decode; bf16 is the top half of fp32).
float half_bits_to_float(uint16_t h) {
  const uint32_t sign = (h >> 15) & 1u, exp = (h >> 10) & 0x1Fu, man = h & 0x3FFu;
  float v;
  if (exp == 0) v = std::ldexp(static_cast<float>(man), -24);
  else if (exp == 31) v = man ? NAN : INFINITY;
  else v = std::ldexp(static_cast<float>(man | 0x400u), static_cast<int>(exp) - 25);
  return sign ? -v : v;
}
float bf16_bits_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// ------------------------------------------------------------------------------ per-device scratch
// Used by the handle-free calls (ns_attn_decode, ns_linear).  Grown on demand, kept until exit.

struct DevScratch {
  void* buf = nullptr;
  size_t bytes = 0;
  int* counters = nullptr;
  size_t n_counters = 0;
  int* err = nullptr;
};
std::mutex g_scratch_mu;
DevScratch g_scratch[64];

ns_status scratch_get(size_t bytes, size_t n_counters, DevScratch** out) {
  int dev = 0;
  NS_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(NS_ERR_UNSUPPORTED, "device index");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  DevScratch& s = g_scratch[dev];
  if (s.err == nullptr) {
    NS_CUDA(cudaMalloc(&s.err, sizeof(int)));
    NS_CUDA(cudaMemset(s.err, 0, sizeof(int)));
  }
  if (s.bytes < bytes) {
    if (s.buf) cudaFree(s.buf);
    s.buf = nullptr;
    s.bytes = 0;
    NS_CUDA(cudaMalloc(&s.buf, bytes));
    s.bytes = bytes;
  }
  if (s.n_counters < n_counters) {
    if (s.counters) cudaFree(s.counters);
    s.counters = nullptr;
    s.n_counters = 0;
    NS_CUDA(cudaMalloc(&s.counters, n_counters * sizeof(int)));
    NS_CUDA(cudaMemset(s.counters, 0, n_counters * sizeof(int)));
    s.n_counters = n_counters;
  }
  *out = &s;
  return NS_OK;
}

}  // namespace

void ns::set_last_error(const char* msg) { g_msg = msg ? msg : ""; }


// ------------------------------------------------------------------------------ block pool

struct ns_block_pool {
  int num_blocks = 0, block_size = 0, mb = 0;
  std::deque<int> free_list;
  std::vector<uint8_t> held;  // 1 while a block is handed out (a block has one owner)

  void reset(int n) {
    num_blocks = n;
    free_list.clear();
    for (int i = 0; i < n; ++i) free_list.push_back(i);
    held.assign(static_cast<size_t>(n), 0);
  }
  int take() {
    const int id = free_list.front();
    free_list.pop_front();
    held[static_cast<size_t>(id)] = 1;
    return id;
  }
};

namespace {

ns_status pool_prepare(ns_block_pool* p, int batch, const int32_t* positions, int32_t* block_tables,
                       int64_t* slot_mapping) {
  if (positions == nullptr || block_tables == nullptr || slot_mapping == nullptr || batch < 0)
    return fail(NS_ERR_INVALID_ARG, "argument");
  const int bs = p->block_size, mb = p->mb;
  size_t need = 0;
  for (int b = 0; b < batch; ++b) {
    const int pos = positions[b];
    if (pos < 0 || pos / bs >= mb) return fail(NS_ERR_INVALID_ARG, "position beyond the block table");
    if (pos % bs == 0) ++need;
  }
  if (need > p->free_list.size()) return fail(NS_ERR_OUT_OF_BLOCKS, "out of KV blocks");
  for (int b = 0; b < batch; ++b) {
    const int pos = positions[b];
    int32_t* row = block_tables + static_cast<size_t>(b) * mb;
    if (pos % bs == 0) row[pos / bs] = p->take();
    slot_mapping[b] = static_cast<int64_t>(row[pos / bs]) * bs + pos % bs;
  }
  return NS_OK;
}

ns_status pool_reserve(ns_block_pool* p, int n, int32_t* out_ids) {
  if ((n > 0 && out_ids == nullptr) || n < 0) return fail(NS_ERR_INVALID_ARG, "argument");
  if (static_cast<size_t>(n) > p->free_list.size()) return fail(NS_ERR_OUT_OF_BLOCKS, "out of KV blocks");
  for (int i = 0; i < n; ++i) out_ids[i] = p->take();
  return NS_OK;
}

ns_status pool_release(ns_block_pool* p, const int32_t* ids, int n) {
  if ((n > 0 && ids == nullptr) || n < 0) return fail(NS_ERR_INVALID_ARG, "argument");
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= p->num_blocks) return fail(NS_ERR_INVALID_ARG, "block id out of range");
  // each id must be handed out and appear once: mark as seen (2), undo the marks on failure
  for (int i = 0; i < n; ++i) {
    uint8_t& h = p->held[static_cast<size_t>(ids[i])];
    if (h != 1) {
      for (int j = 0; j < i; ++j) p->held[static_cast<size_t>(ids[j])] = 1;
      return fail(NS_ERR_INVALID_ARG, "block not in use (already free, or twice in one release)");
    }
    h = 2;
  }
  for (int i = 0; i < n; ++i) {
    p->held[static_cast<size_t>(ids[i])] = 0;
    p->free_list.push_back(ids[i]);
  }
  return NS_OK;
}

ns_status check_meta(int num_blocks, int bs, int mb, int vocab, int max_batch, int batch,
                     const int32_t* token_ids, const int32_t* positions, const int32_t* block_tables,
                     const int32_t* seq_lens, const int64_t* slot_mapping, int src_rows = 0) {
  // src_rows > 0: a device token source of that many rows is set; token ids may then be NULL
  // (row b reads source row b) or -(r + 1) (row b reads source row r < src_rows)
  if (batch < 1 || batch > max_batch) return fail(NS_ERR_INVALID_ARG, "batch out of range");
  if ((src_rows == 0 && !token_ids) || !positions || !block_tables || !seq_lens || !slot_mapping)
    return fail(NS_ERR_INVALID_ARG, "null argument");
  const long long cap = static_cast<long long>(mb) * bs;
  for (int b = 0; b < batch; ++b) {
    const int p = positions[b], L = seq_lens[b];
    if (token_ids && (token_ids[b] >= vocab || token_ids[b] < -src_rows))
      return fail(NS_ERR_INVALID_ARG, "token id out of range");
    // bound the position before p + 1 is formed (no overflow, no table read past the row)
    if (p < 0 || p >= cap) return fail(NS_ERR_INVALID_ARG, "position outside [0, max_blocks_per_seq * block_size)");
    if (L != p + 1) return fail(NS_ERR_INVALID_ARG, "seq_lens must equal positions + 1");
    const int32_t* row = block_tables + static_cast<size_t>(b) * mb;
    const int nblk = (L + bs - 1) / bs;
    for (int i = 0; i < nblk; ++i)
      if (row[i] < 0 || row[i] >= num_blocks) return fail(NS_ERR_INVALID_ARG, "block id out of range");
    if (slot_mapping[b] != static_cast<int64_t>(row[p / bs]) * bs + p % bs)
      return fail(NS_ERR_INVALID_ARG, "slot_mapping disagrees with block_tables");
  }
  return NS_OK;
}

// First rows of the prompt chunks of a step whose metadata passed check_meta: working back from
// the last row, each maximal run of at least kPrefillMinRows rows at consecutive positions that
// read the same blocks as the run's last row is one chunk; the first shorter run ends the search.
std::vector<int> prompt_chunk_starts(int batch, const int32_t* positions, const int32_t* block_tables,
                                     const int32_t* seq_lens, int mb, int bs) {
  std::vector<int> runs;
  int end = batch;
  while (end > 0) {
    const int32_t* tl = block_tables + static_cast<size_t>(end - 1) * mb;
    int f = end - 1;
    while (f > 0) {
      const int b = f - 1;
      if (positions[b] != positions[f] - 1) break;
      const int need = (seq_lens[b] + bs - 1) / bs;
      if (std::memcmp(block_tables + static_cast<size_t>(b) * mb, tl, static_cast<size_t>(need) * 4) != 0) break;
      f = b;
    }
    if (end - f < kPrefillMinRows) break;
    runs.insert(runs.begin(), f);
    end = f;
  }
  return runs;
}

}  // namespace

// ------------------------------------------------------------------------------ the handle

struct Proj {
  void* w = nullptr;
  bool owned = true;
  int N = 0, K = 0, splits = 1, kb_per = 1;
  CUtensorMap mapA;
};

struct LayerDev {
  Proj qkv, o, gu, down;
  float* attn_norm = nullptr;
  float* ffn_norm = nullptr;
};


struct ns_ctx {
  ns_model_cfg cfg;
  int dev = 0, sms = 1, dtype = 0;
  int R = 0;  // activation rows (max_batch)
  std::vector<LayerDev> layers;
  Proj lm;
  void* embed = nullptr;
  float* final_norm = nullptr;
  // activations
  float* resid = nullptr;
  void* xn = nullptr;
  float* sumsq = nullptr;
  void* q = nullptr;
  void* o = nullptr;
  void* act = nullptr;
  float* rope_cos = nullptr;
  float* rope_sin = nullptr;
  double* inv_freq = nullptr;
  std::map<std::tuple<const void*, int>, CUtensorMap> bmaps;
  // KV cache
  int num_blocks = 0, block_size = 0, max_chunks = 1;
  void* pools = nullptr;
  std::vector<void*> kpool, vpool;
  ns_block_pool pool;
  int* attn_counters = nullptr;
  float* attn_partials = nullptr;
  // metadata
  size_t meta_cap = 0;
  uint8_t* meta_host = nullptr;
  uint8_t* meta_dev = nullptr;
  cudaEvent_t meta_done = nullptr;
  bool meta_pending = false;
  // nano-batching
  int n_split = 1;
  std::vector<int> split_sizes;
  int attn_budget = 0;
  int gemm_budget = 0;  // persistent-GEMM CTA cap of nano-batched steps (ns_set_gemm_cta_budget)
  // the decode attention launches of the step being enqueued use the unit-queue variant (set
  // from the step's sequence lengths; part of the graph key)
  bool attn_queue = false;
  std::vector<int> attn_grid_memo;  // attn_max_grid per row count (0: not yet asked)
  std::vector<int> buckets;  // graph batch sizes (ns_set_graph_buckets), ascending
  bool graph_chunks = true;  // steps with prompt chunks replay graphs too (ns_set_graph_chunks)
  int chunk_first = 0;       // rows [chunk_first, batch) of the current step form prefill
                             // chunks (chunk_first == the step's row count: none)
  std::vector<int> chunk_runs;  // first row of each chunk, ascending; a chunk ends where the
                                // next begins (the last at the batch end)
  bool with_lm = true;  // false: the step stops after the last layer (logits_out == NULL)
  const int32_t* tok_src = nullptr;  // device token ids (ns_set_token_source) or null: metadata
  std::vector<uint8_t> dirty_blocks;  // scratch of early_fetch_ok, all zero between calls
  cudaStream_t side = nullptr, cap = nullptr;
  std::vector<cudaEvent_t> events;
  // KV offload: each step's new K/V rows, staged on the device by the QKV epilogues and copied
  // on `copy` to the caller's pinned mirror [n_layers][R][2][kv_dim] (ns_set_kv_offload)
  void* kv_host = nullptr;
  void* kv_stage = nullptr;
  cudaStream_t copy = nullptr;
  // contiguous device buffer and slots of ns_kv_reload / ns_kv_save (grown on demand)
  void* kv_xfer = nullptr;
  size_t kv_xfer_cap = 0;
  long long* kv_slots = nullptr;
  size_t kv_slots_cap = 0;
  // graphs
  struct GraphEntry {
    cudaGraphExec_t ex;
    ns_graph_info info;
  };
  std::map<std::vector<int>, GraphEntry> graphs;
  int* err = nullptr;
  ns_step_info info{};
  int kernels_last = 0;
  // per-kernel timing (eager only)
  bool timing = false;
  // per-tensor trace of one layer (ns_set_trace; eager steps only)
  int trace_layer = -1;
  ns_trace_bufs trace{};
  struct TimedLaunch {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<TimedLaunch> timed;
  ns_kernel_timing timing_acc{};
  // persistent step kernel (ns_set_step_kernel): mode and its device resources
  int step_mode = 0;
  struct StepDev {
    int grid = 0, nslot = 0, max_ch = 1;
    size_t smem = 0, wpack_bytes = 0, sync_bytes = 0;
    StepParams shape{};            // stage tiles, chunks, splits, rotations
    uint8_t* wpack = nullptr;
    long long* streams = nullptr;  // stream_off [grid + 1], then stream_lm [grid]
    float* norms = nullptr;        // attention-norm gains [n_layers][H], then FFN-norm gains
    float* sumsq16 = nullptr;      // [kStepMaxRows][H / 16]
    float* part = nullptr;         // attention partials
    float* split_part = nullptr;   // split-K partial tiles
    unsigned* sync = nullptr;      // barrier word, abort flag, attention and split-K counters
  };
  StepDev* step = nullptr;
};

namespace {

struct MetaLayout {
  size_t tok, pos, seq, slot, tab, logits, flags, total;
};

MetaLayout meta_layout(int B, int MB) {
  MetaLayout m;
  size_t o = 0;
  m.tok = o; o += static_cast<size_t>(B) * 4;
  m.pos = o; o += static_cast<size_t>(B) * 4;
  m.seq = o; o += static_cast<size_t>(B) * 4;
  o = (o + 15) & ~size_t(15);
  m.slot = o; o += static_cast<size_t>(B) * 8;
  m.tab = o; o += static_cast<size_t>(B) * MB * 4;
  o = (o + 15) & ~size_t(15);
  m.logits = o; o += 8;
  m.flags = o; o += 8;  // int early_ok (see AttnParams), int rows_valid (real rows)
  m.total = o;
  return m;
}

enum KernelKind { K_EMBED = 0, K_QKV = 1, K_ATTN = 2, K_O = 3, K_GU = 4, K_DOWN = 5, K_LM = 6 };

// Event pair around one launch when per-kernel timing is on.
struct TimeScope {
  ns_ctx* h;
  cudaStream_t s;
  int kind;
  cudaEvent_t a = nullptr, b = nullptr;
  TimeScope(ns_ctx* h_, cudaStream_t s_, int kind_) : h(h_), s(s_), kind(kind_) {
    if (!h->timing) return;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a, s);
  }
  ~TimeScope() {
    if (!h->timing) return;
    cudaEventRecord(b, s);
    h->timed.push_back({kind, a, b});
  }
};

ns_status get_bmap(ns_ctx* h, const void* buf, int cols, int BN, const CUtensorMap** out) {
  auto key = std::make_tuple(buf, BN);
  auto it = h->bmaps.find(key);
  if (it == h->bmaps.end()) {
    CUtensorMap m;
    NS_TRY(make_tmap(&m, buf, h->dtype, static_cast<uint64_t>(h->R), static_cast<uint64_t>(cols),
                     static_cast<uint32_t>(BN)));
    it = h->bmaps.emplace(key, m).first;
  }
  *out = &it->second;
  return NS_OK;
}

// A handle built for dense batches (its row capacity gives the unsplit weight two 256-token
// output tiles per SM) keeps the weight unsplit: its full batches then run the persistent
// kernel, whose units need no reduction (measured on the 70B-shaped layer at 2048 rows: O 362 ->
// 244 us, down 818 -> 732 us, the unsplit layer 3.69 -> 3.49 ms).  The split stays a function of
// the weight and the handle, never of a launch's rows, so a row's result does not depend on
// the batch it is in.
void choose_splits_for_handle(int N, int K, int R, int sms, int* splits, int* kb_per) {
  choose_splits(N, K, sms, splits, kb_per);
  const long long tiles = static_cast<long long>((R + kMaxBN - 1) / kMaxBN) * (N / kGemmTileN);
  if (tiles >= 2LL * sms) {
    *splits = 1;
    *kb_per = K / kGemmTileK;
  }
}

ns_status init_proj(ns_ctx* h, Proj& p, int N, int K) {
  p.N = N;
  p.K = K;
  choose_splits_for_handle(N, K, h->R, h->sms, &p.splits, &p.kb_per);
  return make_tmap(&p.mapA, p.w, h->dtype, static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                   kGemmTileN);
}

ns_status copy_gain(ns_ctx* h, const void* src, float** dst) {
  const int H = h->cfg.hidden;
  std::vector<uint16_t> raw(H);
  NS_CUDA(cudaMemcpy(raw.data(), src, H * 2, cudaMemcpyDefault));
  std::vector<float> f(H);
  for (int i = 0; i < H; ++i)
    f[i] = h->dtype == NS_BF16 ? bf16_bits_to_float(raw[i]) : half_bits_to_float(raw[i]);
  NS_CUDA(cudaMalloc(dst, H * sizeof(float)));
  NS_CUDA(cudaMemcpy(*dst, f.data(), H * sizeof(float), cudaMemcpyHostToDevice));
  return NS_OK;
}

// Launch parameters of one projection over m rows: the persistent kernel where use_persistent
// says so (its grid in *grid), else the cluster kernel (*grid = 0).
GemmParams proj_params(const Proj& pr, int m, int row0, int epi, int dtype, int sms, int* grid) {
  GemmParams p{};
  p.M = m;
  p.row0 = row0;
  p.N = pr.N;
  p.K = pr.K;
  p.splits = pr.splits;
  p.kb_per_split = pr.kb_per;
  p.epi = epi;
  const int n_tiles = pr.N / kGemmTileN;
  if (use_persistent(m, pr.splits, n_tiles, sms)) {
    p.BN = pick_bn_persistent(m);
    p.tiles_m = (m + p.BN - 1) / p.BN;
    p.nstage = gemm_persistent_stages(p.BN);
    *grid = static_cast<int>(std::min<long long>(static_cast<long long>(p.tiles_m) * n_tiles, sms));
  } else {
    p.BN = pick_bn(m, pr.kb_per, pr.splits, n_tiles, sms);
    p.nstage = gemm_pick_stages(p.BN, p.kb_per_split, ((m + p.BN - 1) / p.BN) * n_tiles, p.splits);
    *grid = 0;
  }
  p.idesc = gemm_idesc(dtype, p.BN);
  return p;
}

ns_status launch_proj(ns_ctx* h, const Proj& pr, const void* x, int x_cols, int row0, int m,
                      int epi, const EpiArgs& e, cudaStream_t s, int kind) {
  int grid = 0;
  GemmParams p = proj_params(pr, m, row0, epi, h->dtype, h->sms, &grid);
  p.err = h->err;
  p.e = e;
  const CUtensorMap* mb = nullptr;
  NS_TRY(get_bmap(h, x, x_cols, p.BN, &mb));
  TimeScope ts(h, s, kind);
  if (grid > 0 && h->n_split > 1 && h->gemm_budget > 0) grid = std::min(grid, h->gemm_budget);
  if (grid > 0) {
    NS_CUDA(launch_gemm_persistent(&pr.mapA, mb, p, h->dtype, grid, s, true));
  } else {
    NS_CUDA(launch_gemm(&pr.mapA, mb, p, h->dtype, s, true));
  }
  h->kernels_last++;
  return NS_OK;
}

void free_step(ns_ctx* h) {
  if (h->step == nullptr) return;
  ns_ctx::StepDev* sd = h->step;
  cudaFree(sd->wpack);
  cudaFree(sd->streams);
  cudaFree(sd->split_part);
  cudaFree(sd->norms);
  cudaFree(sd->sumsq16);
  cudaFree(sd->part);
  cudaFree(sd->sync);
  delete sd;
  h->step = nullptr;
  h->step_mode = 0;
}

// The persistent step kernel takes a step when it is switched on and the step is plain decode
// of at most kStepMaxRows rows on one stream with nothing else to emit.
bool step_kernel_takes(const ns_ctx* h, int B) {
  return h->step_mode == 1 && h->step != nullptr && B <= kStepMaxRows && h->n_split <= 1 &&
         h->chunk_runs.empty() && h->kv_host == nullptr && h->trace_layer < 0 && !h->timing;
}

ns_status enqueue_step_persistent(ns_ctx* h, int B, cudaStream_t s) {
  const ns_model_cfg& c = h->cfg;
  const ns_ctx::StepDev& sd = *h->step;
  const MetaLayout ml = meta_layout(B, c.max_blocks_per_seq);
  StepParams p = sd.shape;
  p.B = B;
  p.H = c.hidden;
  p.d = c.head_dim;
  p.Hq = c.n_q_heads;
  p.Hkv = c.n_kv_heads;
  p.G = c.n_q_heads / c.n_kv_heads;
  p.qd = c.n_q_heads * c.head_dim;
  p.kvd = c.n_kv_heads * c.head_dim;
  p.F = c.ffn;
  p.vocab = c.vocab;
  p.n_layers = c.n_layers;
  p.eps = c.rms_eps;
  p.scale_log2 = static_cast<float>(1.0 / std::sqrt(static_cast<double>(c.head_dim)) * 1.4426950408889634);
  p.nslot = sd.nslot;
  p.with_lm = h->with_lm ? 1 : 0;
  p.wpack = sd.wpack;
  p.stream_off = sd.streams;
  p.stream_lm = sd.streams + sd.grid + 1;
  p.embed = h->embed;
  p.attn_norm = sd.norms;
  p.ffn_norm = sd.norms + static_cast<size_t>(c.n_layers) * c.hidden;
  p.final_norm = h->final_norm;
  p.pools = static_cast<uint8_t*>(h->pools);
  p.pool_bytes = static_cast<size_t>(static_cast<uint8_t*>(h->vpool[0]) - static_cast<uint8_t*>(h->kpool[0]));
  p.num_blocks = h->num_blocks + 1;  // + padding block
  p.mb = c.max_blocks_per_seq;
  p.block_size = h->block_size;
  p.pool_slots = static_cast<long long>(h->num_blocks + 1) * h->block_size;
  p.tok = reinterpret_cast<const int*>(h->meta_dev + ml.tok);
  p.tok_src = h->tok_src;
  p.pos = reinterpret_cast<const int*>(h->meta_dev + ml.pos);
  p.seq = reinterpret_cast<const int*>(h->meta_dev + ml.seq);
  p.slot = reinterpret_cast<const long long*>(h->meta_dev + ml.slot);
  p.tab = reinterpret_cast<const int*>(h->meta_dev + ml.tab);
  p.logits_slot = reinterpret_cast<const unsigned long long*>(h->meta_dev + ml.logits);
  p.rows_valid = reinterpret_cast<const int*>(h->meta_dev + ml.flags) + 1;
  p.early_ok = reinterpret_cast<const int*>(h->meta_dev + ml.flags);
  p.inv_freq = h->inv_freq;
  p.resid = h->resid;
  p.xn = h->xn;
  p.q = h->q;
  p.o = h->o;
  p.act = h->act;
  p.sumsq16 = sd.sumsq16;
  p.split_part = sd.split_part;
  p.attn_part = sd.part;
  p.max_ch = sd.max_ch;
  p.sync = sd.sync;
  p.err = h->err;
  NS_CUDA(cudaMemsetAsync(sd.sync, 0, sd.sync_bytes, s));
  NS_CUDA(launch_step(p, h->dtype, sd.grid, sd.smem, s));
  h->kernels_last = 1;
  return NS_OK;
}

// Grid of a decode attention launch over `rows` rows: one full wave (memoised per row count),
// at most one CTA per unit, within the attention CTA budget.
int attn_grid(ns_ctx* h, int rows) {
  const ns_model_cfg& c = h->cfg;
  if (static_cast<int>(h->attn_grid_memo.size()) <= rows) h->attn_grid_memo.resize(rows + 1, 0);
  int& wave = h->attn_grid_memo[rows];
  if (wave == 0) wave = attn_max_grid(h->dtype, c.head_dim, c.n_q_heads / c.n_kv_heads, rows);
  int grid = std::min(wave, rows * c.n_kv_heads * h->max_chunks);
  if (h->attn_budget > 0) grid = std::min(grid, h->attn_budget);
  return std::max(grid, 1);
}

// Whether a step over B rows launches the unit-queue variant of decode attention: when the
// decode rows of some nano-batch hold at least kAttnQueueUnits (row, kv head, superchunk) units
// per CTA of its launch.  seq: the step's host sequence lengths (B of them); null takes the
// most any row could hold.
bool attn_queue_for(ns_ctx* h, int B, const int32_t* seq) {
  const int Hkv = h->cfg.n_kv_heads;
  int r = 0;
  const int n = h->n_split <= 1 ? 1 : h->n_split;
  for (int i = 0; i < n; ++i) {
    const int rows = h->n_split <= 1 ? B : h->split_sizes[i];
    const int r_lo = r, r_hi = r + rows;
    r = r_hi;
    const int d_hi = std::min(r_hi, std::max(r_lo, h->chunk_first));
    if (d_hi <= r_lo) continue;
    long long chunks = 0;
    for (int b = r_lo; b < d_hi; ++b)
      chunks += seq != nullptr ? attn_num_chunks(seq[b]) : h->max_chunks;
    if (chunks * Hkv >= static_cast<long long>(kAttnQueueUnits) * attn_grid(h, d_hi - r_lo))
      return true;
  }
  return false;
}

// Enqueue one step for `B` rows on `s0` (and the side stream when nano-batched).
ns_status enqueue_step(ns_ctx* h, int B, cudaStream_t s0) {
  if (step_kernel_takes(h, B)) return enqueue_step_persistent(h, B, s0);
  const ns_model_cfg& c = h->cfg;
  const int H = c.hidden, d = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, F = c.ffn;
  const int qd = Hq * d, kvd = Hkv * d;
  const MetaLayout ml = meta_layout(B, c.max_blocks_per_seq);
  const int* m_tok = reinterpret_cast<const int*>(h->meta_dev + ml.tok);
  const int* m_pos = reinterpret_cast<const int*>(h->meta_dev + ml.pos);
  const int* m_seq = reinterpret_cast<const int*>(h->meta_dev + ml.seq);
  const long long* m_slot = reinterpret_cast<const long long*>(h->meta_dev + ml.slot);
  const int* m_tab = reinterpret_cast<const int*>(h->meta_dev + ml.tab);
  const unsigned long long* m_logits = reinterpret_cast<const unsigned long long*>(h->meta_dev + ml.logits);
  const int* m_rows_valid = reinterpret_cast<const int*>(h->meta_dev + ml.flags) + 1;
  h->kernels_last = 0;

  // nano-batches: (row0, rows)
  std::vector<std::pair<int, int>> nb;
  if (h->n_split <= 1) {
    nb.push_back({0, B});
  } else {
    int r = 0;
    for (int i = 0; i < h->n_split; ++i) {
      nb.push_back({r, h->split_sizes[i]});
      r += h->split_sizes[i];
    }
  }
  const int n = static_cast<int>(nb.size());
  cudaStream_t st[2] = {s0, h->side};
  // events: fork, side-stream join, copy-stream join, and per (layer, nano-batch) QKV completion
  const bool mirror = h->kv_host != nullptr;
  const size_t kv_row_bytes = static_cast<size_t>(2) * kvd * 2;
  auto ev_qkv = [&](int l, int i) { return h->events[3 + static_cast<size_t>(l) * n + i]; };
  const size_t need_ev = 3 + static_cast<size_t>(c.n_layers) * n;
  while (h->events.size() < need_ev) {
    cudaEvent_t ev;
    NS_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    h->events.push_back(ev);
  }
  if (n > 1) {
    NS_CUDA(cudaEventRecord(h->events[0], s0));
    NS_CUDA(cudaStreamWaitEvent(h->side, h->events[0], 0));
  }
  const int G = Hq / Hkv;
  const float scale_log2 = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)) * 1.4426950408889634);

  // rows [row0, row0 + rows) of a [R][row_bytes] activation buffer to a trace buffer
  auto trace_copy = [&](int l, void* dst, const void* src, size_t row_bytes, int row0, int rows,
                        cudaStream_t s) -> cudaError_t {
    if (l != h->trace_layer || dst == nullptr) return cudaSuccess;
    const size_t off = static_cast<size_t>(row0) * row_bytes;
    return cudaMemcpyAsync(static_cast<uint8_t*>(dst) + off, static_cast<const uint8_t*>(src) + off,
                           static_cast<size_t>(rows) * row_bytes, cudaMemcpyDeviceToDevice, s);
  };
  const size_t q_row_bytes = static_cast<size_t>(qd) * 2, r_row_bytes = static_cast<size_t>(H) * 4;

  EpiArgs norm{};  // common fused-RMSNorm inputs
  norm.sumsq_in = h->sumsq;
  norm.sumsq_tiles = H / kGemmTileN;
  norm.sumsq_ld = h->R;
  norm.norm_dim = H;
  norm.eps = c.rms_eps;

  for (int i = 0; i < n; ++i) {
    EmbedParams ep{};
    ep.embed = h->embed;
    ep.token_ids = m_tok;
    ep.tok_src = h->tok_src;
    ep.rows_valid = m_rows_valid;
    ep.positions = m_pos;
    ep.vocab = c.vocab;
    ep.hidden = H;
    ep.gamma = h->layers[0].attn_norm;
    ep.resid = h->resid;
    ep.xn = h->xn;
    ep.sumsq = h->sumsq;
    ep.sumsq_ld = h->R;
    ep.rope_cos = h->rope_cos;
    ep.rope_sin = h->rope_sin;
    ep.head_dim = d;
    ep.inv_freq = h->inv_freq;
    ep.batch = nb[i].second;
    ep.row0 = nb[i].first;
    ep.err = h->err;
    {
      TimeScope ts(h, st[i % 2], K_EMBED);
      NS_CUDA(launch_embed(ep, h->dtype, st[i % 2], true));
    }
    h->kernels_last++;
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerDev& L = h->layers[l];
    for (int i = 0; i < n; ++i) {
      EpiArgs e = norm;
      e.q_out = h->q;
      e.k_pool = h->kpool[l];
      e.v_pool = h->vpool[l];
      e.slot_mapping = m_slot;
      e.rope_cos = h->rope_cos;
      e.rope_sin = h->rope_sin;
      e.q_dim = qd;
      e.kv_dim = kvd;
      e.head_dim = d;
      e.n_kv_heads = Hkv;
      e.block_size = h->block_size;
      e.pool_slots = static_cast<long long>(h->num_blocks + 1) * h->block_size;  // + padding block
      e.kv_stage = mirror ? static_cast<uint8_t*>(h->kv_stage) + static_cast<size_t>(l) * h->R * kv_row_bytes
                          : nullptr;
      NS_TRY(launch_proj(h, L.qkv, h->xn, H, nb[i].first, nb[i].second, EPI_QKV, e,
                         st[i % 2], K_QKV));
      NS_CUDA(trace_copy(l, h->trace.q, h->q, q_row_bytes, nb[i].first, nb[i].second, st[i % 2]));
      if (n > 1 || mirror) NS_CUDA(cudaEventRecord(ev_qkv(l, i), st[i % 2]));
      if (mirror) {
        // the rows' K/V leave for the host while attention and the FFN of this layer run
        NS_CUDA(cudaStreamWaitEvent(h->copy, ev_qkv(l, i), 0));
        const size_t off = (static_cast<size_t>(l) * h->R + nb[i].first) * kv_row_bytes;
        NS_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(h->kv_host) + off,
                                static_cast<uint8_t*>(h->kv_stage) + off,
                                static_cast<size_t>(nb[i].second) * kv_row_bytes, cudaMemcpyDeviceToHost,
                                h->copy));
      }
    }
    for (int i = 0; i < n; ++i) {
      cudaStream_t s = st[i % 2];
      for (int j = 0; j < i; ++j)
        if ((j % 2) != (i % 2)) NS_CUDA(cudaStreamWaitEvent(s, ev_qkv(l, j), 0));
      AttnParams ap{};
      ap.q = h->q;
      ap.q_row_stride = qd;
      ap.k_pool = h->kpool[l];
      ap.v_pool = h->vpool[l];
      ap.block_tables = m_tab;
      ap.mb = c.max_blocks_per_seq;
      ap.seq_lens = m_seq;
      ap.out = h->o;
      ap.out_row_stride = qd;
      ap.batch = nb[i].second;
      ap.row0 = nb[i].first;
      ap.n_kv_heads = Hkv;
      ap.num_blocks = h->num_blocks + 1;  // + padding block
      ap.block_size = h->block_size;
      ap.scale_log2 = scale_log2;
      ap.max_chunks = h->max_chunks;
      ap.partials = h->attn_partials;
      ap.counters = h->attn_counters;
      ap.sched = reinterpret_cast<unsigned*>(h->attn_counters + static_cast<size_t>(h->R) * Hkv) +
                 nb[i].first;
      ap.err = h->err;
      ap.early_ok = reinterpret_cast<const int*>(h->meta_dev + ml.flags);
      // decode rows of the nano-batch, then the prefill-chunk rows it holds (chunks come last)
      const int r_lo = nb[i].first, r_hi = nb[i].first + nb[i].second;
      const int d_hi = std::min(r_hi, std::max(r_lo, h->chunk_first));
      if (d_hi > r_lo) {
        ap.batch = d_hi - r_lo;
        const int grid = attn_grid(h, ap.batch);
        TimeScope ts(h, s, K_ATTN);
        NS_CUDA(launch_attn(ap, h->dtype, d, G, grid, s, true, h->attn_queue));
        h->kernels_last++;
      }
      for (size_t ci = 0; ci < h->chunk_runs.size(); ++ci) {
        // the part of chunk [c_lo, c_hi) inside this nano-batch
        const int c_lo = h->chunk_runs[ci];
        const int c_hi = ci + 1 < h->chunk_runs.size() ? h->chunk_runs[ci + 1] : B;
        const int p_lo = std::max(c_lo, r_lo), p_hi = std::min(c_hi, r_hi);
        if (p_hi <= p_lo) continue;
        PrefillParams pp{};
        pp.q = h->q;
        pp.q_row_stride = qd;
        pp.k_pool = h->kpool[l];
        pp.v_pool = h->vpool[l];
        pp.block_tables = m_tab;
        pp.mb = c.max_blocks_per_seq;
        pp.table_row = c_hi - 1;
        pp.positions = m_pos;
        pp.out = h->o;
        pp.out_row_stride = qd;
        pp.row0 = p_lo;
        pp.chunk = p_hi - p_lo;
        pp.n_kv_heads = Hkv;
        pp.num_blocks = h->num_blocks + 1;
        pp.scale_log2 = scale_log2;
        pp.err = h->err;
        TimeScope ts(h, s, K_ATTN);
        NS_CUDA(launch_prefill(pp, h->dtype, d, G, s, true));
        h->kernels_last++;
      }

      NS_CUDA(trace_copy(l, h->trace.attn, h->o, q_row_bytes, r_lo, r_hi - r_lo, s));

      EpiArgs eo{};
      eo.resid = h->resid;
      eo.xn_out = h->xn;
      eo.gamma_next = L.ffn_norm;
      eo.sumsq_out = h->sumsq;
      eo.sumsq_ld = h->R;
      eo.resid_dim = H;
      NS_TRY(launch_proj(h, L.o, h->o, qd, nb[i].first, nb[i].second, EPI_RESID, eo, s, K_O));
      NS_CUDA(trace_copy(l, h->trace.resid_mid, h->resid, r_row_bytes, r_lo, r_hi - r_lo, s));

      EpiArgs eg = norm;
      eg.act_out = h->act;
      eg.ffn = F;
      NS_TRY(launch_proj(h, L.gu, h->xn, H, nb[i].first, nb[i].second, EPI_SWIGLU, eg, s, K_GU));

      EpiArgs ed{};
      ed.resid = h->resid;
      ed.xn_out = h->xn;
      ed.gamma_next = (l + 1 < c.n_layers) ? h->layers[l + 1].attn_norm : h->final_norm;
      ed.sumsq_out = h->sumsq;
      ed.sumsq_ld = h->R;
      ed.resid_dim = H;
      NS_TRY(launch_proj(h, L.down, h->act, F, nb[i].first, nb[i].second, EPI_RESID, ed, s, K_DOWN));
      NS_CUDA(trace_copy(l, h->trace.resid_out, h->resid, r_row_bytes, r_lo, r_hi - r_lo, s));
    }
  }
  for (int i = 0; i < n && h->with_lm; ++i) {
    EpiArgs el = norm;
    el.out_ptr_slot = m_logits;
    el.rows_valid = m_rows_valid;
    el.ldo = c.vocab;
    NS_TRY(launch_proj(h, h->lm, h->xn, H, nb[i].first, nb[i].second, EPI_F32, el,
                       st[i % 2], K_LM));
  }
  if (n > 1) {
    NS_CUDA(cudaEventRecord(h->events[1], h->side));
    NS_CUDA(cudaStreamWaitEvent(s0, h->events[1], 0));
  }
  if (mirror) {  // the step completes when its K/V are on the host
    NS_CUDA(cudaEventRecord(h->events[2], h->copy));
    NS_CUDA(cudaStreamWaitEvent(s0, h->events[2], 0));
  }
  return NS_OK;
}

// True when no row reads, at a block other than its last, a block that this step writes (the
// block of some row's slot).  Decode-only batches satisfy it; rows of a prefill chunk sharing
// one block table do not.  The metadata has passed check_meta.
bool early_fetch_ok(ns_ctx* h, int batch, const int32_t* block_tables, const int32_t* seq_lens,
                    const int64_t* slot_mapping) {
  const int bs = h->block_size, mb = h->cfg.max_blocks_per_seq;
  std::vector<uint8_t>& dirty = h->dirty_blocks;
  if (dirty.size() != static_cast<size_t>(h->num_blocks)) dirty.assign(h->num_blocks, 0);
  for (int b = 0; b < batch; ++b) dirty[slot_mapping[b] / bs] = 1;
  bool ok = true;
  for (int b = 0; b < batch && ok; ++b) {
    const int nbk = (seq_lens[b] + bs - 1) / bs;
    const int32_t* row = block_tables + static_cast<size_t>(b) * mb;
    for (int j = 0; j + 1 < nbk; ++j)
      if (dirty[row[j]]) {
        ok = false;
        break;
      }
  }
  for (int b = 0; b < batch; ++b) dirty[slot_mapping[b] / bs] = 0;
  return ok;
}

std::vector<int> graph_key(const ns_ctx* h, int B) {
  const uint64_t src = reinterpret_cast<uint64_t>(h->tok_src);
  const uint64_t kvh = reinterpret_cast<uint64_t>(h->kv_host);
  std::vector<int> k{B, h->step_mode, h->n_split, h->attn_budget, h->n_split > 1 ? h->gemm_budget : 0, h->with_lm ? 1 : 0,
                     static_cast<int>(src & 0xffffffffu), static_cast<int>(src >> 32),
                     h->chunk_first, static_cast<int>(kvh & 0xffffffffu), static_cast<int>(kvh >> 32),
                     static_cast<int>(h->chunk_runs.size()), h->attn_queue ? 1 : 0};
  for (int v : h->chunk_runs) k.push_back(v);
  for (int v : h->split_sizes) k.push_back(v);
  return k;
}

ns_status get_graph(ns_ctx* h, int B, cudaGraphExec_t* out) {
  auto key = graph_key(h, B);
  auto it = h->graphs.find(key);
  if (it != h->graphs.end()) {
    *out = it->second.ex;
    return NS_OK;
  }
  const auto t0 = std::chrono::steady_clock::now();
  NS_CUDA(cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal));
  ns_status st = enqueue_step(h, B, h->cap);
  cudaGraph_t g = nullptr;
  cudaError_t ce = cudaStreamEndCapture(h->cap, &g);
  if (st != NS_OK) {
    if (g) cudaGraphDestroy(g);
    return st;
  }
  if (ce != cudaSuccess) return fail(NS_ERR_CUDA, std::string("graph capture: ") + cudaGetErrorString(ce));
  cudaGraphExec_t ex = nullptr;
  ce = cudaGraphInstantiate(&ex, g, 0);
  size_t n_nodes = 0;
  cudaGraphGetNodes(g, nullptr, &n_nodes);
  std::vector<cudaGraphNode_t> nodes(n_nodes);
  int kernels = 0;
  if (n_nodes) {
    cudaGraphGetNodes(g, nodes.data(), &n_nodes);
    for (auto nd : nodes) {
      cudaGraphNodeType t;
      if (cudaGraphNodeGetType(nd, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++kernels;
    }
  }
  cudaGraphDestroy(g);
  if (ce != cudaSuccess) return fail(NS_ERR_CUDA, std::string("graph instantiate: ") + cudaGetErrorString(ce));
  ns_graph_info gi{};
  gi.batch = B;
  gi.n_split = h->n_split;
  gi.attn_cta_budget = h->attn_budget;
  gi.gemm_cta_budget = h->n_split > 1 ? h->gemm_budget : 0;
  gi.attn_queue = h->attn_queue ? 1 : 0;
  gi.with_lm = h->with_lm ? 1 : 0;
  gi.chunk_rows = h->chunk_first < B ? B - h->chunk_first : 0;
  gi.kv_offload = h->kv_host != nullptr ? 1 : 0;
  gi.kernels = kernels;
  gi.capture_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  h->graphs.emplace(key, ns_ctx::GraphEntry{ex, gi});
  h->info.graphs_cached = static_cast<int>(h->graphs.size());
  h->info.kernels_per_step = kernels;
  h->info.last_capture_ms = gi.capture_ms;
  *out = ex;
  return NS_OK;
}

void free_proj(Proj& p) {
  if (p.owned && p.w) cudaFree(p.w);
  p.w = nullptr;
}

}  // namespace

// ================================================================================== C ABI

extern "C" {

const char* ns_status_str(ns_status s) {
  switch (s) {
    case NS_OK: return "NS_OK";
    case NS_ERR_INVALID_ARG: return "NS_ERR_INVALID_ARG";
    case NS_ERR_OUT_OF_MEMORY: return "NS_ERR_OUT_OF_MEMORY";
    case NS_ERR_CUDA: return "NS_ERR_CUDA";
    case NS_ERR_UNSUPPORTED: return "NS_ERR_UNSUPPORTED";
    case NS_ERR_NOT_INITIALIZED: return "NS_ERR_NOT_INITIALIZED";
    case NS_ERR_DEVICE_CHECK: return "NS_ERR_DEVICE_CHECK";
    case NS_ERR_OUT_OF_BLOCKS: return "NS_ERR_OUT_OF_BLOCKS";
  }
  return "NS_ERR_UNKNOWN";
}

const char* ns_last_error_message(void) { return g_msg.c_str(); }

void ns_destroy(ns_handle h) {
  if (h == nullptr) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->dev);
  cudaDeviceSynchronize();
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second.ex);
  for (auto& L : h->layers) {
    free_proj(L.qkv);
    free_proj(L.o);
    free_proj(L.gu);
    free_proj(L.down);
    cudaFree(L.attn_norm);
    cudaFree(L.ffn_norm);
  }
  free_proj(h->lm);
  cudaFree(h->embed);
  cudaFree(h->final_norm);
  cudaFree(h->resid);
  cudaFree(h->xn);
  cudaFree(h->sumsq);
  cudaFree(h->q);
  cudaFree(h->o);
  cudaFree(h->act);
  cudaFree(h->rope_cos);
  cudaFree(h->rope_sin);
  cudaFree(h->inv_freq);
  cudaFree(h->pools);
  cudaFree(h->attn_counters);
  cudaFree(h->attn_partials);
  free_step(h);
  cudaFreeHost(h->meta_host);
  cudaFree(h->meta_dev);
  cudaFree(h->err);
  if (h->meta_done) cudaEventDestroy(h->meta_done);
  for (auto ev : h->events) cudaEventDestroy(ev);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->cap) cudaStreamDestroy(h->cap);
  if (h->copy) cudaStreamDestroy(h->copy);
  cudaFree(h->kv_stage);
  cudaFree(h->kv_xfer);
  cudaFree(h->kv_slots);
  delete h;
  cudaSetDevice(prev);
}

ns_status ns_create(const ns_model_cfg* cfg, const ns_weights* w, ns_handle* out) {
  if (cfg == nullptr || w == nullptr || out == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const ns_model_cfg& c = *cfg;
  if (c.hidden <= 0 || c.n_layers <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 ||
      c.ffn <= 0 || c.vocab <= 0 || c.max_batch <= 0 || c.max_blocks_per_seq <= 0 ||
      c.n_q_heads % c.n_kv_heads != 0 || !(c.rms_eps >= 0.f) || !(c.rope_theta > 0.0))
    return fail(NS_ERR_INVALID_ARG, "model dims");
  if (c.dtype != NS_F16 && c.dtype != NS_BF16) return fail(NS_ERR_INVALID_ARG, "dtype");
  if (c.max_batch > kMaxRows) return fail(NS_ERR_UNSUPPORTED, "max_batch above 4096");
  if (c.max_blocks_per_seq > 4096) return fail(NS_ERR_UNSUPPORTED, "max_blocks_per_seq above 4096");
  const int H = c.hidden, d = c.head_dim, qd = c.n_q_heads * d, kvd = c.n_kv_heads * d, F = c.ffn;
  const int G = c.n_q_heads / c.n_kv_heads;
  if (H % 128 || qd % 128 || kvd % 128 || (2 * F) % 128 || c.vocab % 128 || F % 64 ||
      !attn_supported(d, G, 16) || c.vocab / kGemmTileN > 65535 || (2 * F) / kGemmTileN > 65535)
    return fail(NS_ERR_UNSUPPORTED, "shape not implemented (see ns.h)");
  if (w->embed == nullptr || w->final_norm == nullptr || w->layers == nullptr ||
      (!c.tie_embeddings && w->lm_head == nullptr))
    return fail(NS_ERR_INVALID_ARG, "weight pointers");
  for (int l = 0; l < c.n_layers; ++l) {
    const ns_layer_weights& lw = w->layers[l];
    if (!lw.attn_norm || !lw.wq || !lw.wk || !lw.wv || !lw.wo || !lw.ffn_norm || !lw.w_gate ||
        !lw.w_up || !lw.w_down)
      return fail(NS_ERR_INVALID_ARG, "layer weight pointers");
  }
  ns_ctx* h = new ns_ctx();
  h->cfg = c;
  h->dtype = c.dtype;
  h->R = c.max_batch;
  cudaGetDevice(&h->dev);
  h->sms = device_sms();
  auto bail = [&](ns_status s) {
    std::string keep = g_msg;
    ns_destroy(h);
    g_msg = keep;
    return s;
  };
#define CK(expr)                       \
  do {                                 \
    ns_status s__ = (expr);            \
    if (s__ != NS_OK) return bail(s__); \
  } while (0)
  auto cuda = [&](cudaError_t e, const char* what) -> ns_status {
    if (e == cudaSuccess) return NS_OK;
    return fail(e == cudaErrorMemoryAllocation ? NS_ERR_OUT_OF_MEMORY : NS_ERR_CUDA,
                std::string(what) + ": " + cudaGetErrorString(e));
  };
  const size_t e2 = 2;
  h->layers.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    const ns_layer_weights& lw = w->layers[l];
    LayerDev& L = h->layers[l];
    // QKV concatenated: rows q | k | v
    CK(cuda(cudaMalloc(&L.qkv.w, static_cast<size_t>(qd + 2 * kvd) * H * e2), "malloc qkv"));
    uint8_t* q8 = static_cast<uint8_t*>(L.qkv.w);
    CK(cuda(cudaMemcpy(q8, lw.wq, static_cast<size_t>(qd) * H * e2, cudaMemcpyDefault), "copy wq"));
    CK(cuda(cudaMemcpy(q8 + static_cast<size_t>(qd) * H * e2, lw.wk, static_cast<size_t>(kvd) * H * e2,
                       cudaMemcpyDefault), "copy wk"));
    CK(cuda(cudaMemcpy(q8 + static_cast<size_t>(qd + kvd) * H * e2, lw.wv,
                       static_cast<size_t>(kvd) * H * e2, cudaMemcpyDefault), "copy wv"));
    CK(init_proj(h, L.qkv, qd + 2 * kvd, H));
    CK(cuda(cudaMalloc(&L.o.w, static_cast<size_t>(H) * qd * e2), "malloc wo"));
    CK(cuda(cudaMemcpy(L.o.w, lw.wo, static_cast<size_t>(H) * qd * e2, cudaMemcpyDefault), "copy wo"));
    CK(init_proj(h, L.o, H, qd));
    // gate/up interleaved in 64-row groups: [gate 64j..64j+63 ; up 64j..64j+63] per 128 rows
    CK(cuda(cudaMalloc(&L.gu.w, static_cast<size_t>(2 * F) * H * e2), "malloc gate/up"));
    const size_t grp = static_cast<size_t>(64) * H * e2;
    CK(cuda(cudaMemcpy2D(L.gu.w, 2 * grp, lw.w_gate, grp, grp, F / 64, cudaMemcpyDefault), "copy gate"));
    CK(cuda(cudaMemcpy2D(static_cast<uint8_t*>(L.gu.w) + grp, 2 * grp, lw.w_up, grp, grp, F / 64,
                         cudaMemcpyDefault), "copy up"));
    CK(init_proj(h, L.gu, 2 * F, H));
    CK(cuda(cudaMalloc(&L.down.w, static_cast<size_t>(H) * F * e2), "malloc down"));
    CK(cuda(cudaMemcpy(L.down.w, lw.w_down, static_cast<size_t>(H) * F * e2, cudaMemcpyDefault), "copy down"));
    CK(init_proj(h, L.down, H, F));
    CK(copy_gain(h, lw.attn_norm, &L.attn_norm));
    CK(copy_gain(h, lw.ffn_norm, &L.ffn_norm));
  }
  CK(cuda(cudaMalloc(&h->embed, static_cast<size_t>(c.vocab) * H * e2), "malloc embed"));
  CK(cuda(cudaMemcpy(h->embed, w->embed, static_cast<size_t>(c.vocab) * H * e2, cudaMemcpyDefault), "copy embed"));
  CK(copy_gain(h, w->final_norm, &h->final_norm));
  if (c.tie_embeddings) {
    h->lm.w = h->embed;
    h->lm.owned = false;
  } else {
    CK(cuda(cudaMalloc(&h->lm.w, static_cast<size_t>(c.vocab) * H * e2), "malloc lm_head"));
    CK(cuda(cudaMemcpy(h->lm.w, w->lm_head, static_cast<size_t>(c.vocab) * H * e2, cudaMemcpyDefault),
            "copy lm_head"));
  }
  CK(init_proj(h, h->lm, c.vocab, H));
  // activations
  const size_t R = h->R;
  CK(cuda(cudaMalloc(&h->resid, R * H * 4), "malloc resid"));
  CK(cuda(cudaMalloc(&h->xn, R * H * e2), "malloc xn"));
  CK(cuda(cudaMalloc(&h->sumsq, R * (H / 128) * 4), "malloc sumsq"));
  CK(cuda(cudaMalloc(&h->q, R * qd * e2), "malloc q"));
  CK(cuda(cudaMalloc(&h->o, R * qd * e2), "malloc o"));
  CK(cuda(cudaMalloc(&h->act, R * F * e2), "malloc act"));
  CK(cuda(cudaMalloc(&h->rope_cos, R * (d / 2) * 4), "malloc rope"));
  CK(cuda(cudaMalloc(&h->rope_sin, R * (d / 2) * 4), "malloc rope"));
  {
    // RoPE inverse frequencies theta^(-2i/d), computed once on the host in fp64
    std::vector<double> inv(d / 2);
    for (int i = 0; i < d / 2; ++i) inv[i] = std::pow(c.rope_theta, -2.0 * i / static_cast<double>(d));
    CK(cuda(cudaMalloc(&h->inv_freq, inv.size() * sizeof(double)), "malloc inv_freq"));
    CK(cuda(cudaMemcpy(h->inv_freq, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice),
            "copy inv_freq"));
  }
  CK(cuda(cudaMemset(h->xn, 0, R * H * e2), "memset"));
  CK(cuda(cudaMemset(h->o, 0, R * qd * e2), "memset"));
  CK(cuda(cudaMemset(h->act, 0, R * F * e2), "memset"));
  // metadata: pinned host staging + device copy, sized for max_batch
  h->meta_cap = meta_layout(h->R, c.max_blocks_per_seq).total;
  CK(cuda(cudaMallocHost(&h->meta_host, h->meta_cap), "pinned metadata"));
  CK(cuda(cudaMalloc(&h->meta_dev, h->meta_cap), "metadata"));
  CK(cuda(cudaEventCreateWithFlags(&h->meta_done, cudaEventDisableTiming), "event"));
  CK(cuda(cudaMalloc(&h->err, sizeof(int)), "err"));
  CK(cuda(cudaMemset(h->err, 0, sizeof(int)), "err"));
  CK(cuda(cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking), "stream"));
  CK(cuda(cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking), "stream"));
  CK(cuda(cudaDeviceSynchronize(), "create sync"));
#undef CK
  *out = h;
  return NS_OK;
}

ns_status ns_kv_alloc(ns_handle h, int num_blocks, int block_size) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (h->pools != nullptr) return fail(NS_ERR_INVALID_ARG, "KV pools already allocated");
  if (num_blocks <= 0 || block_size != 16)
    return fail(num_blocks <= 0 ? NS_ERR_INVALID_ARG : NS_ERR_UNSUPPORTED, "num_blocks > 0, block_size 16");
  const ns_model_cfg& c = h->cfg;
  // one block past the caller's pool takes the rows that pad a batch up to a graph bucket
  const long long blocks = static_cast<long long>(num_blocks) + 1;
  const long long pool_rows = blocks * c.n_kv_heads * block_size;
  if (pool_rows >= (1ll << 31))
    return fail(NS_ERR_UNSUPPORTED, "pool rows (blocks * kv heads * block_size) must fit in int32");
  const size_t pool = static_cast<size_t>(pool_rows) * c.head_dim * 2;
  NS_CUDA(cudaSetDevice(h->dev));
  NS_CUDA(cudaMalloc(&h->pools, pool * 2 * c.n_layers));
  // never-written slots read as zeros (finite), never as stale garbage
  NS_CUDA(cudaMemset(h->pools, 0, pool * 2 * c.n_layers));
  h->kpool.resize(c.n_layers);
  h->vpool.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    h->kpool[l] = static_cast<uint8_t*>(h->pools) + pool * (2 * static_cast<size_t>(l));
    h->vpool[l] = static_cast<uint8_t*>(h->pools) + pool * (2 * static_cast<size_t>(l) + 1);
  }
  h->num_blocks = num_blocks;
  h->block_size = block_size;
  h->max_chunks = attn_max_chunks(c.max_blocks_per_seq * block_size);
  const int G = c.n_q_heads / c.n_kv_heads;
  const size_t rows_heads = static_cast<size_t>(h->R) * c.n_kv_heads;
  // superchunk counters [R][n_kv_heads], then a unit-queue counter per possible first row of an
  // attention launch (nano-batches on two streams run concurrently)
  NS_CUDA(cudaMalloc(&h->attn_counters, (rows_heads + h->R) * sizeof(int)));
  NS_CUDA(cudaMemset(h->attn_counters, 0, (rows_heads + h->R) * sizeof(int)));
  NS_CUDA(cudaMalloc(&h->attn_partials,
                     rows_heads * attn_slot_floats(h->max_chunks, G, c.head_dim) * sizeof(float)));
  h->pool.block_size = block_size;
  h->pool.mb = c.max_blocks_per_seq;
  h->pool.reset(num_blocks);
  return NS_OK;
}

ns_status ns_kv_layer_ptrs(ns_handle h, int layer, void** k_pool, void** v_pool) {
  if (h == nullptr || k_pool == nullptr || v_pool == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  if (h->pools == nullptr) return fail(NS_ERR_NOT_INITIALIZED, "ns_kv_alloc first");
  if (layer < 0 || layer >= h->cfg.n_layers) return fail(NS_ERR_INVALID_ARG, "layer");
  *k_pool = h->kpool[layer];
  *v_pool = h->vpool[layer];
  return NS_OK;
}

ns_status ns_kv_prepare_step(ns_handle h, int batch, const int32_t* positions, int32_t* block_tables,
                             int64_t* slot_mapping) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (h->pools == nullptr) return fail(NS_ERR_NOT_INITIALIZED, "ns_kv_alloc first");
  return pool_prepare(&h->pool, batch, positions, block_tables, slot_mapping);
}

ns_status ns_kv_reserve(ns_handle h, int n, int32_t* out_ids) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (h->pools == nullptr) return fail(NS_ERR_NOT_INITIALIZED, "ns_kv_alloc first");
  return pool_reserve(&h->pool, n, out_ids);
}

ns_status ns_kv_release(ns_handle h, const int32_t* block_ids, int n) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (h->pools == nullptr) return fail(NS_ERR_NOT_INITIALIZED, "ns_kv_alloc first");
  return pool_release(&h->pool, block_ids, n);
}

ns_status ns_kv_free_count(ns_handle h, int* n_free) {
  if (h == nullptr || n_free == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  *n_free = static_cast<int>(h->pool.free_list.size());
  return NS_OK;
}

ns_status ns_pool_create(int num_blocks, int block_size, int max_blocks_per_seq, ns_pool* out) {
  if (out == nullptr || num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0)
    return fail(NS_ERR_INVALID_ARG, "pool arguments");
  ns_block_pool* p = new ns_block_pool();
  p->block_size = block_size;
  p->mb = max_blocks_per_seq;
  p->reset(num_blocks);
  *out = p;
  return NS_OK;
}

void ns_pool_destroy(ns_pool p) { delete p; }

ns_status ns_pool_prepare_step(ns_pool p, int batch, const int32_t* positions, int32_t* block_tables,
                               int64_t* slot_mapping) {
  if (p == nullptr) return fail(NS_ERR_INVALID_ARG, "null pool");
  return pool_prepare(p, batch, positions, block_tables, slot_mapping);
}

ns_status ns_pool_reserve(ns_pool p, int n, int32_t* out_ids) {
  if (p == nullptr) return fail(NS_ERR_INVALID_ARG, "null pool");
  return pool_reserve(p, n, out_ids);
}

ns_status ns_pool_release(ns_pool p, const int32_t* block_ids, int n) {
  if (p == nullptr) return fail(NS_ERR_INVALID_ARG, "null pool");
  return pool_release(p, block_ids, n);
}

ns_status ns_pool_geometry(ns_pool p, int* num_blocks, int* block_size) {
  if (p == nullptr || num_blocks == nullptr || block_size == nullptr)
    return fail(NS_ERR_INVALID_ARG, "null argument");
  *num_blocks = p->num_blocks;
  *block_size = p->block_size;
  return NS_OK;
}

ns_status ns_kv_get_pool(ns_handle h, ns_pool* out) {
  if (h == nullptr || out == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  if (h->pools == nullptr) return fail(NS_ERR_NOT_INITIALIZED, "ns_kv_alloc first");
  *out = &h->pool;
  return NS_OK;
}

ns_status ns_pool_free_count(ns_pool p, int* n_free) {
  if (p == nullptr || n_free == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  *n_free = static_cast<int>(p->free_list.size());
  return NS_OK;
}

ns_status ns_check_step_metadata(int num_blocks, int block_size, int max_blocks_per_seq, int vocab,
                                 int max_batch, int batch, const int32_t* token_ids,
                                 const int32_t* positions, const int32_t* block_tables,
                                 const int32_t* seq_lens, const int64_t* slot_mapping) {
  if (num_blocks < 1 || block_size < 1 || max_blocks_per_seq < 1 || vocab < 1)
    return fail(NS_ERR_INVALID_ARG, "pool arguments");
  return check_meta(num_blocks, block_size, max_blocks_per_seq, vocab, max_batch, batch, token_ids,
                    positions, block_tables, seq_lens, slot_mapping);
}

ns_status ns_find_prompt_chunks(int block_size, int max_blocks_per_seq, int batch,
                                const int32_t* positions, const int32_t* block_tables,
                                const int32_t* seq_lens, int32_t* starts, int capacity, int* n) {
  if (n == nullptr || (batch > 0 && (!positions || !block_tables || !seq_lens)) ||
      (capacity > 0 && starts == nullptr))
    return fail(NS_ERR_INVALID_ARG, "null argument");
  if (block_size < 1 || max_blocks_per_seq < 1 || batch < 0 || capacity < 0)
    return fail(NS_ERR_INVALID_ARG, "block_size, max_blocks_per_seq >= 1; batch, capacity >= 0");
  const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] < 1 || seq_lens[b] > cap || positions[b] < 0)
      return fail(NS_ERR_INVALID_ARG, "seq_len outside [1, max_blocks_per_seq * block_size] or a negative position");
  const std::vector<int> runs =
      prompt_chunk_starts(batch, positions, block_tables, seq_lens, max_blocks_per_seq, block_size);
  *n = static_cast<int>(runs.size());
  for (int i = 0; i < std::min(*n, capacity); ++i) starts[i] = runs[static_cast<size_t>(i)];
  return NS_OK;
}

ns_status ns_set_nanobatch(ns_handle h, int n_split, const int* sizes, int attn_cta_budget) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (n_split < 1 || n_split > 4) return fail(NS_ERR_INVALID_ARG, "n_split must be 1..4");
  std::vector<int> s;
  if (n_split > 1) {
    if (sizes == nullptr) return fail(NS_ERR_INVALID_ARG, "sizes required for n_split > 1");
    for (int i = 0; i < n_split; ++i) {
      if (sizes[i] <= 0) return fail(NS_ERR_INVALID_ARG, "nano-batch sizes must be positive");
      s.push_back(sizes[i]);
    }
  }
  h->n_split = n_split;
  h->split_sizes = s;
  h->attn_budget = attn_cta_budget > 0 ? attn_cta_budget : 0;
  return NS_OK;
}

ns_status ns_set_step_kernel(ns_handle h, int mode) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (mode != 0 && mode != 1) return fail(NS_ERR_INVALID_ARG, "mode must be 0 or 1");
  if (mode == 0 || h->step != nullptr) {
    h->step_mode = mode;
    return NS_OK;
  }
  const ns_model_cfg& c = h->cfg;
  const int H = c.hidden, d = c.head_dim, F = c.ffn, G = c.n_q_heads / c.n_kv_heads;
  const int qd = c.n_q_heads * d, kvd = c.n_kv_heads * d;
  if ((d != 64 && d != 128) || G > 8 || F % 128 != 0 || H > 4096)
    return fail(NS_ERR_UNSUPPORTED, "persistent step: head_dim 64 or 128, at most 8 query heads per KV head, ffn a multiple of 128, hidden at most 4096");
  NS_CUDA(cudaSetDevice(h->dev));
  int smem_max = 0;
  NS_CUDA(cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev));
  const long long room = static_cast<long long>(smem_max) - static_cast<long long>(step_smem_bytes(d, 0));
  const int nslot = static_cast<int>(room / (kStepSlot + 16));
  if (nslot < 4) return fail(NS_ERR_UNSUPPORTED, "persistent step: too little shared memory");
  const size_t smem = step_smem_bytes(d, nslot);
  int per_sm = 0;
  NS_CUDA(step_configure(h->dtype, d, smem, &per_sm));
  if (per_sm < 1) return fail(NS_ERR_UNSUPPORTED, "persistent step: kernel does not fit an SM");
  const int grid = h->sms;
  // per stage: 16-row output tiles, 128-column chunks of the reduction, K splits (reductions
  // longer than kStepSliceChunks chunks), round-robin start of unsplit stages (each stage
  // continues where the previous one stopped, spreading a layer's tiles over the SMs)
  StepParams sh{};
  sh.n_layers = c.n_layers;
  sh.n_tiles[SS_QKV] = (qd + 2 * kvd) / 16;
  sh.kc[SS_QKV] = H / 128;
  sh.n_tiles[SS_O] = H / 16;
  sh.kc[SS_O] = qd / 128;
  sh.n_tiles[SS_GU] = F / 8;
  sh.kc[SS_GU] = H / 128;
  sh.n_tiles[SS_DOWN] = H / 16;
  sh.kc[SS_DOWN] = F / 128;
  sh.n_tiles[SS_LM] = c.vocab / 16;
  sh.kc[SS_LM] = H / 128;
  int rot = 0;
  for (int k = 0; k < SS_COUNT; ++k) {
    sh.split[k] = (sh.kc[k] + kStepSliceChunks - 1) / kStepSliceChunks;
    sh.rot[k] = k == SS_LM ? 0 : rot % grid;
    if (k != SS_LM && sh.split[k] == 1) rot += sh.n_tiles[k];
    if (sh.split[k] > 1) sh.max_split_tiles = std::max(sh.max_split_tiles, sh.n_tiles[k]);
  }
  StepPlan plan;
  if (!build_step_plan(grid, sh, &plan))
    return fail(NS_ERR_UNSUPPORTED, "persistent step: a reduction needs more than 8 splits or a CTA more than 32 split tiles");
  // the chunk stream of every CTA, in the order its compute warps consume it
  const long long n_chunks = plan.stream_off[grid];
  std::vector<PackDesc> desc;
  desc.reserve(static_cast<size_t>(n_chunks));
  const int nrope = (c.n_q_heads + c.n_kv_heads) * (d / 16);
  auto emit = [&](int k, const StepTiles& t, int l) {
    for (int g0 = 0; g0 < t.count; g0 += kStepGroup) {
      const int tg = std::min(kStepGroup, t.count - g0);
      for (int kc = t.kc0; kc < t.kc1; ++kc)
        for (int ti = 0; ti < tg; ++ti) {
          const int tile = t.first + (g0 + ti) * t.stride;
          PackDesc pd{};
          pd.kc = kc;
          pd.tile = tile;
          pd.kind = PK_PLAIN;
          pd.row0 = tile * 16;
          if (k == SS_QKV) {
            pd.w = h->layers[l].qkv.w;
            pd.K = H;
            if (tile < nrope) {
              pd.kind = PK_ROPE;
            } else {
              pd.row0 = qd + kvd + (tile - nrope) * 16;
            }
          } else if (k == SS_O) {
            pd.w = h->layers[l].o.w;
            pd.K = qd;
          } else if (k == SS_GU) {
            pd.w = h->layers[l].gu.w;
            pd.K = H;
            pd.kind = PK_GU;
          } else if (k == SS_DOWN) {
            pd.w = h->layers[l].down.w;
            pd.K = F;
          } else {
            pd.w = h->lm.w;
            pd.K = H;
          }
          desc.push_back(pd);
        }
    }
  };
  for (int cta = 0; cta < grid; ++cta) {
    for (int l = 0; l < c.n_layers; ++l)
      for (int k : {SS_QKV, SS_O, SS_GU, SS_DOWN})
        emit(k, step_tiles(grid, cta, sh.n_tiles[k], sh.kc[k], sh.split[k], sh.rot[k]), l);
    emit(SS_LM, step_tiles(grid, cta, sh.n_tiles[SS_LM], sh.kc[SS_LM], sh.split[SS_LM], sh.rot[SS_LM]), 0);
  }
  if (static_cast<long long>(desc.size()) != n_chunks)
    return fail(NS_ERR_CUDA, "persistent step: chunk plan inconsistent");
  auto* sd = new ns_ctx::StepDev();
  sd->grid = grid;
  sd->nslot = nslot;
  sd->smem = smem;
  sd->max_ch = (c.max_blocks_per_seq + kStepAttnBlocks - 1) / kStepAttnBlocks;
  sd->wpack_bytes = static_cast<size_t>(n_chunks) * kStepChunk;
  sd->shape = sh;
  sd->sync_bytes = (2 + static_cast<size_t>(c.n_layers) * kStepMaxRows * c.n_kv_heads +
                    (static_cast<size_t>(c.n_layers) + 1) * 4 * sh.max_split_tiles) * sizeof(unsigned);
  h->step = sd;
  auto cuda = [&](cudaError_t e, const char* what) -> ns_status {
    if (e == cudaSuccess) return NS_OK;
    free_step(h);
    return fail(e == cudaErrorMemoryAllocation ? NS_ERR_OUT_OF_MEMORY : NS_ERR_CUDA,
                std::string("persistent step: ") + what + ": " + cudaGetErrorString(e));
  };
  NS_TRY(cuda(cudaMalloc(&sd->wpack, sd->wpack_bytes), "weights"));
  PackDesc* ddesc = nullptr;
  NS_TRY(cuda(cudaMalloc(&ddesc, desc.size() * sizeof(PackDesc)), "pack descriptors"));
  cudaError_t e = cudaMemcpy(ddesc, desc.data(), desc.size() * sizeof(PackDesc), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = launch_step_pack(ddesc, n_chunks, sd->wpack, d, nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  cudaFree(ddesc);
  NS_TRY(cuda(e, "pack"));
  NS_TRY(cuda(cudaMalloc(&sd->streams, (2 * static_cast<size_t>(grid) + 1) * sizeof(long long)), "plan"));
  NS_TRY(cuda(cudaMemcpy(sd->streams, plan.stream_off.data(), (grid + 1) * sizeof(long long), cudaMemcpyHostToDevice), "plan"));
  NS_TRY(cuda(cudaMemcpy(sd->streams + grid + 1, plan.stream_lm.data(), grid * sizeof(long long), cudaMemcpyHostToDevice), "plan"));
  size_t split_floats = 16;
  for (int k = 0; k < SS_COUNT; ++k)
    if (sh.split[k] > 1)
      split_floats = std::max(split_floats, static_cast<size_t>(sh.n_tiles[k]) * sh.split[k] * kStepMaxRows * 16);
  NS_TRY(cuda(cudaMalloc(&sd->split_part, split_floats * sizeof(float)), "split partials"));
  NS_TRY(cuda(cudaMalloc(&sd->norms, 2 * static_cast<size_t>(c.n_layers) * H * sizeof(float)), "norms"));
  for (int l = 0; l < c.n_layers; ++l) {
    NS_TRY(cuda(cudaMemcpy(sd->norms + static_cast<size_t>(l) * H, h->layers[l].attn_norm, H * sizeof(float),
                           cudaMemcpyDeviceToDevice), "norms"));
    NS_TRY(cuda(cudaMemcpy(sd->norms + (static_cast<size_t>(c.n_layers) + l) * H, h->layers[l].ffn_norm,
                           H * sizeof(float), cudaMemcpyDeviceToDevice), "norms"));
  }
  NS_TRY(cuda(cudaMalloc(&sd->sumsq16, static_cast<size_t>(H / 16) * kStepMaxRows * sizeof(float)), "sums"));
  NS_TRY(cuda(cudaMemset(sd->sumsq16, 0, static_cast<size_t>(H / 16) * kStepMaxRows * sizeof(float)), "sums"));
  const size_t part = static_cast<size_t>(kStepMaxRows) * c.n_kv_heads * sd->max_ch * G * (d + 2);
  NS_TRY(cuda(cudaMalloc(&sd->part, part * sizeof(float)), "attention partials"));
  NS_TRY(cuda(cudaMalloc(&sd->sync, sd->sync_bytes), "sync"));
  NS_TRY(cuda(cudaMemset(sd->sync, 0, sd->sync_bytes), "sync"));
  h->step_mode = 1;
  return NS_OK;
}

ns_status ns_set_gemm_cta_budget(ns_handle h, int gemm_cta_budget) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (gemm_cta_budget < 0) return fail(NS_ERR_INVALID_ARG, "gemm_cta_budget < 0");
  h->gemm_budget = gemm_cta_budget;
  return NS_OK;
}

ns_status ns_decode_step(ns_handle h, int batch, const int32_t* token_ids, const int32_t* positions,
                         const int32_t* block_tables, const int32_t* seq_lens,
                         const int64_t* slot_mapping, float* logits_out, ns_stream_t stream) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (h->pools == nullptr) return fail(NS_ERR_NOT_INITIALIZED, "ns_kv_alloc first");
  const ns_model_cfg& c = h->cfg;
  const int bs = h->block_size, mb = c.max_blocks_per_seq;
  const int src_rows = h->tok_src != nullptr ? h->R : 0;
  NS_TRY(check_meta(h->num_blocks, bs, mb, c.vocab, c.max_batch, batch, token_ids, positions,
                    block_tables, seq_lens, slot_mapping, src_rows));
  if (h->n_split > 1) {
    int sum = 0;
    for (int v : h->split_sizes) sum += v;
    if (sum != batch) return fail(NS_ERR_INVALID_ARG, "nano-batch sizes do not sum to the batch");
  }
  NS_CUDA(cudaSetDevice(h->dev));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // one packed metadata buffer, one host-to-device copy
  if (h->meta_pending) NS_CUDA(cudaEventSynchronize(h->meta_done));
  // prefill chunks, each attended by one causal kernel (the rows before them are decode rows)
  std::vector<int> runs = prompt_chunk_starts(batch, positions, block_tables, seq_lens, mb, bs);
  bool graphed = c.use_graphs && !h->timing && h->trace_layer < 0;
  if (graphed && !h->graph_chunks && !runs.empty()) graphed = false;  // layouts vary: eager
  // graph batch: the smallest bucket that holds the rows; padding rows fill the rest, and a
  // padded step has no chunk layout (its chunk rows, if any, use the decode kernel)
  int Bg = batch;
  if (graphed && h->n_split <= 1)
    for (int v : h->buckets)
      if (v >= batch) {
        Bg = v;
        break;
      }
  if (Bg != batch) runs.clear();
  h->chunk_runs = runs;
  h->chunk_first = runs.empty() ? Bg : runs.front();  // Bg: none, so padded steps share a graph
  const MetaLayout ml = meta_layout(Bg, mb);
  uint8_t* mh = h->meta_host;
  if (token_ids != nullptr) {
    std::memcpy(mh + ml.tok, token_ids, batch * 4);
  } else {  // every row reads its own row of the device token source
    int32_t* t = reinterpret_cast<int32_t*>(mh + ml.tok);
    for (int b = 0; b < batch; ++b) t[b] = -(b + 1);
  }
  std::memcpy(mh + ml.pos, positions, batch * 4);
  std::memcpy(mh + ml.seq, seq_lens, batch * 4);
  std::memcpy(mh + ml.slot, slot_mapping, batch * 8);
  std::memcpy(mh + ml.tab, block_tables, static_cast<size_t>(batch) * mb * 4);
  // padding rows: token 0 at position 0 in the padding block (past the caller's pool)
  const int pad_block = h->num_blocks;
  for (int b = batch; b < Bg; ++b) {
    const int32_t zero = 0, one = 1;
    const int64_t slot = static_cast<int64_t>(pad_block) * bs;
    std::memcpy(mh + ml.tok + b * 4, &zero, 4);
    std::memcpy(mh + ml.pos + b * 4, &zero, 4);
    std::memcpy(mh + ml.seq + b * 4, &one, 4);
    std::memcpy(mh + ml.slot + b * 8, &slot, 8);
    int32_t* row = reinterpret_cast<int32_t*>(mh + ml.tab) + static_cast<size_t>(b) * mb;
    std::memset(row, 0, static_cast<size_t>(mb) * 4);
    row[0] = pad_block;
  }
  const unsigned long long lp = reinterpret_cast<unsigned long long>(logits_out);
  std::memcpy(mh + ml.logits, &lp, 8);
  const int flags[2] = {early_fetch_ok(h, batch, block_tables, seq_lens, slot_mapping) ? 1 : 0,
                        batch};
  std::memcpy(mh + ml.flags, flags, 8);
  NS_CUDA(cudaMemcpyAsync(h->meta_dev, mh, ml.total, cudaMemcpyHostToDevice, s));
  NS_CUDA(cudaEventRecord(h->meta_done, s));
  h->meta_pending = true;
  h->with_lm = logits_out != nullptr;
  h->attn_queue = attn_queue_for(h, graphed ? Bg : batch, reinterpret_cast<const int32_t*>(mh + ml.seq));
  if (graphed) {
    cudaGraphExec_t ex = nullptr;
    NS_TRY(get_graph(h, Bg, &ex));
    NS_CUDA(cudaGraphLaunch(ex, s));
  } else {
    NS_TRY(enqueue_step(h, batch, s));
    h->info.kernels_per_step = h->kernels_last;
  }
  h->info.steps++;
  return NS_OK;
}

ns_status ns_set_graph_buckets(ns_handle h, int n, const int* sizes) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (n < 0 || n > 64 || (n > 0 && sizes == nullptr)) return fail(NS_ERR_INVALID_ARG, "bucket count");
  std::vector<int> v(sizes, sizes + n);
  for (int i = 0; i < n; ++i)
    if (v[i] < 1 || v[i] > h->cfg.max_batch || (i > 0 && v[i] <= v[i - 1]))
      return fail(NS_ERR_INVALID_ARG, "bucket sizes must ascend within [1, max_batch]");
  h->buckets = v;
  return NS_OK;
}

ns_status ns_capture_graphs(ns_handle h, int n, const int* batch_sizes, int with_lm) {
  if (h == nullptr || (n > 0 && batch_sizes == nullptr) || n < 0) return fail(NS_ERR_INVALID_ARG, "argument");
  if (h->pools == nullptr) return fail(NS_ERR_NOT_INITIALIZED, "ns_kv_alloc first");
  if (!h->cfg.use_graphs) return fail(NS_ERR_INVALID_ARG, "the handle does not use graphs");
  int split_sum = 0;
  for (int v : h->split_sizes) split_sum += v;
  for (int i = 0; i < n; ++i) {
    const int B = batch_sizes[i];
    if (B < 1 || B > h->R) return fail(NS_ERR_INVALID_ARG, "batch size outside [1, max_batch]");
    if (h->n_split > 1 && B != split_sum)
      return fail(NS_ERR_INVALID_ARG, "with nano-batches only their total batch is captured");
  }
  NS_CUDA(cudaSetDevice(h->dev));
  for (int i = 0; i < n; ++i) {
    h->with_lm = with_lm != 0;
    h->chunk_first = batch_sizes[i];  // decode-only layout
    h->chunk_runs.clear();
    cudaGraphExec_t ex = nullptr;
    // the fixed-deal attention, and the unit-queue one where the rows could need it
    h->attn_queue = false;
    NS_TRY(get_graph(h, batch_sizes[i], &ex));
    if (attn_queue_for(h, batch_sizes[i], nullptr)) {
      h->attn_queue = true;
      NS_TRY(get_graph(h, batch_sizes[i], &ex));
    }
  }
  return NS_OK;
}

ns_status ns_get_graph_report(ns_handle h, ns_graph_info* out, int capacity, int* n) {
  if (h == nullptr || n == nullptr || (capacity > 0 && out == nullptr)) return fail(NS_ERR_INVALID_ARG, "argument");
  int i = 0;
  for (const auto& kv : h->graphs) {
    if (i < capacity) out[i] = kv.second.info;
    ++i;
  }
  *n = i;
  return NS_OK;
}

ns_status ns_set_graph_chunks(ns_handle h, int capture) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  h->graph_chunks = capture != 0;
  return NS_OK;
}

ns_status ns_set_token_source(ns_handle h, const int32_t* device_token_ids) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  h->tok_src = device_token_ids;
  return NS_OK;
}

ns_status ns_set_kv_offload(ns_handle h, void* host_dst, size_t bytes) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (host_dst == nullptr) {
    h->kv_host = nullptr;
    return NS_OK;
  }
  const ns_model_cfg& c = h->cfg;
  const size_t need = static_cast<size_t>(c.n_layers) * h->R * 2 * c.n_kv_heads * c.head_dim * 2;
  if (bytes < need) return fail(NS_ERR_INVALID_ARG, "host buffer smaller than n_layers * max_batch * 2 * kv_dim elements");
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host_dst) != cudaSuccess || a.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return fail(NS_ERR_INVALID_ARG, "host_dst must be pinned host memory (cudaMallocHost / cudaHostRegister)");
  }
  NS_CUDA(cudaSetDevice(h->dev));
  if (h->kv_stage == nullptr) {
    NS_CUDA(cudaMalloc(&h->kv_stage, need));
    NS_CUDA(cudaMemset(h->kv_stage, 0, need));
  }
  if (h->copy == nullptr) NS_CUDA(cudaStreamCreateWithFlags(&h->copy, cudaStreamNonBlocking));
  h->kv_host = host_dst;
  return NS_OK;
}

namespace {

// Slots of tokens first_pos .. first_pos + n - 1 of one request, uploaded to the handle's slot
// buffer on `s`, and the contiguous transfer buffer grown to `bytes`.
ns_status kv_transfer_setup(ns_ctx* h, int n_tokens, int first_pos, const int32_t* block_table, int n_table,
                            size_t bytes, cudaStream_t s) {
  if (h->pools == nullptr) return fail(NS_ERR_NOT_INITIALIZED, "ns_kv_alloc first");
  if (n_tokens < 1 || first_pos < 0 || block_table == nullptr || n_table < 1)
    return fail(NS_ERR_INVALID_ARG, "n_tokens >= 1, first_pos >= 0, a block table");
  const int bs = h->block_size;
  const long long last = static_cast<long long>(first_pos) + n_tokens - 1;
  if (last / bs >= n_table) return fail(NS_ERR_INVALID_ARG, "block table shorter than the token range");
  std::vector<long long> slots(n_tokens);
  for (int t = 0; t < n_tokens; ++t) {
    const long long pos = static_cast<long long>(first_pos) + t;
    const int b = block_table[pos / bs];
    if (b < 0 || b >= h->num_blocks) return fail(NS_ERR_INVALID_ARG, "block id out of range");
    slots[t] = static_cast<long long>(b) * bs + pos % bs;
  }
  NS_CUDA(cudaSetDevice(h->dev));
  if (h->kv_xfer_cap < bytes || h->kv_slots_cap < slots.size() * sizeof(long long)) {
    NS_CUDA(cudaDeviceSynchronize());  // earlier transfers may still use the old buffers
    if (h->kv_xfer_cap < bytes) {
      cudaFree(h->kv_xfer);
      h->kv_xfer = nullptr;
      h->kv_xfer_cap = 0;
      NS_CUDA(cudaMalloc(&h->kv_xfer, bytes));
      h->kv_xfer_cap = bytes;
    }
    if (h->kv_slots_cap < slots.size() * sizeof(long long)) {
      cudaFree(h->kv_slots);
      h->kv_slots = nullptr;
      h->kv_slots_cap = 0;
      NS_CUDA(cudaMalloc(&h->kv_slots, slots.size() * sizeof(long long)));
      h->kv_slots_cap = slots.size() * sizeof(long long);
    }
  }
  // pageable source: the call returns once the slots are staged, so `slots` may go
  NS_CUDA(cudaMemcpyAsync(h->kv_slots, slots.data(), slots.size() * sizeof(long long),
                          cudaMemcpyHostToDevice, s));
  return NS_OK;
}

KvCopyParams kv_copy_params(ns_ctx* h, int n_tokens, int to_pool) {
  const ns_model_cfg& c = h->cfg;
  KvCopyParams p{};
  p.pools = h->pools;
  p.pool_bytes = static_cast<size_t>(h->num_blocks + 1) * c.n_kv_heads * h->block_size * c.head_dim * 2;
  p.buf = h->kv_xfer;
  p.slots = h->kv_slots;
  p.n = n_tokens;
  p.n_layers = c.n_layers;
  p.n_kv_heads = c.n_kv_heads;
  p.head_dim = c.head_dim;
  p.block_size = h->block_size;
  p.pool_slots = static_cast<long long>(h->num_blocks) * h->block_size;
  p.to_pool = to_pool;
  p.err = h->err;
  return p;
}

}  // namespace

ns_status ns_kv_reload(ns_handle h, const void* host_src, int n_tokens, int first_pos, const int32_t* block_table,
                       int n_table, ns_stream_t stream) {
  if (h == nullptr || host_src == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  const ns_model_cfg& c = h->cfg;
  const size_t bytes = static_cast<size_t>(c.n_layers) * n_tokens * 2 * c.n_kv_heads * c.head_dim * 2;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  NS_TRY(kv_transfer_setup(h, n_tokens, first_pos, block_table, n_table, bytes, s));
  NS_CUDA(cudaMemcpyAsync(h->kv_xfer, host_src, bytes, cudaMemcpyHostToDevice, s));
  NS_CUDA(launch_kv_copy(kv_copy_params(h, n_tokens, 1), h->sms, s));
  return NS_OK;
}

ns_status ns_kv_save(ns_handle h, void* host_dst, int n_tokens, int first_pos, const int32_t* block_table,
                     int n_table, ns_stream_t stream) {
  if (h == nullptr || host_dst == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  const ns_model_cfg& c = h->cfg;
  const size_t bytes = static_cast<size_t>(c.n_layers) * n_tokens * 2 * c.n_kv_heads * c.head_dim * 2;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  NS_TRY(kv_transfer_setup(h, n_tokens, first_pos, block_table, n_table, bytes, s));
  NS_CUDA(launch_kv_copy(kv_copy_params(h, n_tokens, 0), h->sms, s));
  NS_CUDA(cudaMemcpyAsync(host_dst, h->kv_xfer, bytes, cudaMemcpyDeviceToHost, s));
  return NS_OK;
}

ns_status ns_set_trace(ns_handle h, int layer, const ns_trace_bufs* bufs) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  if (layer >= h->cfg.n_layers) return fail(NS_ERR_INVALID_ARG, "trace layer past the last layer");
  if (layer < 0 || bufs == nullptr) {
    h->trace_layer = -1;
    h->trace = ns_trace_bufs{};
    return NS_OK;
  }
  h->trace_layer = layer;
  h->trace = *bufs;
  return NS_OK;
}

ns_status ns_set_kernel_timing(ns_handle h, int on) {
  if (h == nullptr) return fail(NS_ERR_INVALID_ARG, "null handle");
  h->timing = on != 0;
  return NS_OK;
}

ns_status ns_get_kernel_timing(ns_handle h, ns_kernel_timing* out) {
  if (h == nullptr || out == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  NS_CUDA(cudaSetDevice(h->dev));
  NS_CUDA(cudaDeviceSynchronize());
  for (auto& t : h->timed) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess && t.kind >= 0 && t.kind < NS_KERNEL_KINDS) {
      h->timing_acc.launches[t.kind]++;
      h->timing_acc.total_ms[t.kind] += ms;
    }
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  h->timed.clear();
  *out = h->timing_acc;
  h->timing_acc = ns_kernel_timing{};
  return NS_OK;
}

ns_status ns_get_step_info(ns_handle h, ns_step_info* out) {
  if (h == nullptr || out == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  *out = h->info;
  return NS_OK;
}

ns_status ns_get_device_error(ns_handle h, int* code) {
  if (code == nullptr) return fail(NS_ERR_INVALID_ARG, "null argument");
  int* word = nullptr;
  int* counters = nullptr;  // attention counters a wait that ran out may have left set
  size_t n_counters = 0;
  if (h != nullptr) {
    NS_CUDA(cudaSetDevice(h->dev));
    word = h->err;
    if (h->attn_counters != nullptr) {
      counters = h->attn_counters;
      n_counters = static_cast<size_t>(h->R) * h->cfg.n_kv_heads + h->R;
    }
  } else {
    DevScratch* sc = nullptr;
    NS_TRY(scratch_get(0, 0, &sc));
    word = sc->err;
    counters = sc->counters;
    n_counters = sc->n_counters;
  }
  NS_CUDA(cudaDeviceSynchronize());
  NS_CUDA(cudaMemcpy(code, word, sizeof(int), cudaMemcpyDeviceToHost));
  NS_CUDA(cudaMemset(word, 0, sizeof(int)));
  // a kernel that gave up a wait may not have brought its split-K arrival counters or its unit
  // queue's ticket counter back to zero; no kernel runs now, so clear them for the next launch
  if (*code == NS_DEV_WAIT_TIMEOUT && counters != nullptr && n_counters > 0)
    NS_CUDA(cudaMemset(counters, 0, n_counters * sizeof(int)));
  return NS_OK;
}

ns_status ns_attn_decode(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                         const int32_t* seq_lens, void* out, int batch, int n_q_heads, int n_kv_heads,
                         int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                         int dtype, ns_stream_t stream) {
  return ns_attn_decode_capped(q, k_pool, v_pool, block_tables, seq_lens, out, batch, n_q_heads, n_kv_heads,
                               head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, 0, stream);
}

ns_status ns_attn_decode_capped(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                                const int32_t* seq_lens, void* out, int batch, int n_q_heads, int n_kv_heads,
                                int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                                int dtype, int cta_budget, ns_stream_t stream) {
  if (cta_budget < 0) return fail(NS_ERR_INVALID_ARG, "cta_budget < 0");
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return fail(NS_ERR_INVALID_ARG, "null argument");
  if (batch < 1 || batch > kMaxRows || n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads ||
      max_blocks_per_seq < 1 || num_blocks < 1 || !(scale > 0.f) || (dtype != NS_F16 && dtype != NS_BF16))
    return fail(NS_ERR_INVALID_ARG, "attention arguments");
  const int G = n_q_heads / n_kv_heads;
  if (!attn_supported(head_dim, G, block_size)) return fail(NS_ERR_UNSUPPORTED, "attention shape");
  if (max_blocks_per_seq * block_size > 65536)
    return fail(NS_ERR_UNSUPPORTED, "max_blocks_per_seq * block_size above 65536");
  const int max_chunks = attn_max_chunks(max_blocks_per_seq * block_size);
  const size_t rows_heads = static_cast<size_t>(batch) * n_kv_heads;
  if (static_cast<long long>(num_blocks) * n_kv_heads * block_size >= (1ll << 31))
    return fail(NS_ERR_UNSUPPORTED, "num_blocks * n_kv_heads * block_size must fit in int32");
  DevScratch* sc = nullptr;
  NS_TRY(scratch_get(rows_heads * attn_slot_floats(max_chunks, G, head_dim) * sizeof(float), rows_heads + 1, &sc));
  AttnParams ap{};
  ap.q = q;
  ap.q_row_stride = static_cast<long long>(n_q_heads) * head_dim;
  ap.k_pool = k_pool;
  ap.v_pool = v_pool;
  ap.block_tables = block_tables;
  ap.mb = max_blocks_per_seq;
  ap.seq_lens = seq_lens;
  ap.out = out;
  ap.out_row_stride = static_cast<long long>(n_q_heads) * head_dim;
  ap.batch = batch;
  ap.row0 = 0;
  ap.n_kv_heads = n_kv_heads;
  ap.num_blocks = num_blocks;
  ap.block_size = block_size;
  ap.scale_log2 = scale * 1.4426950408889634f;
  ap.max_chunks = max_chunks;
  ap.partials = static_cast<float*>(sc->buf);
  ap.counters = sc->counters;
  ap.sched = reinterpret_cast<unsigned*>(sc->counters + rows_heads);
  ap.err = sc->err;
  const int cap = attn_max_grid(dtype, head_dim, G, batch);
  const long long units = static_cast<long long>(batch) * n_kv_heads * max_chunks;
  int grid = static_cast<int>(std::min<long long>(cap, units));
  if (cta_budget > 0) grid = std::min(grid, cta_budget);
  // seq_lens are on the device: the queue variant whenever the rows could hold enough units
  // (it falls back to the fixed deal itself when they do not)
  const bool queue = units >= static_cast<long long>(kAttnQueueUnits) * grid;
  NS_CUDA(launch_attn(ap, dtype, head_dim, G, grid, reinterpret_cast<cudaStream_t>(stream), false,
                      queue));
  return NS_OK;
}

ns_status ns_linear(const void* w, const void* x, float* y, int m, int n, int k, int dtype, ns_stream_t stream) {
  if (!w || !x || !y) return fail(NS_ERR_INVALID_ARG, "null argument");
  if (m < 1 || m > kMaxRows || n < 128 || k < 64 || (dtype != NS_F16 && dtype != NS_BF16))
    return fail(NS_ERR_INVALID_ARG, "linear arguments");
  if (n % 128 || k % 64) return fail(NS_ERR_UNSUPPORTED, "n % 128 and k % 64 must be 0");
  if (n / kGemmTileN > 65535) return fail(NS_ERR_UNSUPPORTED, "n above 65535 * 128");
  Proj pr;
  pr.w = const_cast<void*>(w);
  pr.owned = false;
  pr.N = n;
  pr.K = k;
  const int sms = device_sms();
  choose_splits(n, k, sms, &pr.splits, &pr.kb_per);
  NS_TRY(make_tmap(&pr.mapA, w, dtype, static_cast<uint64_t>(n), static_cast<uint64_t>(k), kGemmTileN));
  int grid = 0;
  GemmParams p = proj_params(pr, m, 0, EPI_F32, dtype, sms, &grid);
  DevScratch* sc = nullptr;
  NS_TRY(scratch_get(0, 0, &sc));
  p.err = sc->err;
  p.e.out_f32 = y;
  p.e.ldo = n;
  CUtensorMap mb;
  NS_TRY(make_tmap(&mb, x, dtype, static_cast<uint64_t>(m), static_cast<uint64_t>(k), static_cast<uint32_t>(p.BN)));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (grid > 0) {
    NS_CUDA(launch_gemm_persistent(&pr.mapA, &mb, p, dtype, grid, st, false));
  } else {
    NS_CUDA(launch_gemm(&pr.mapA, &mb, p, dtype, st, false));
  }
  return NS_OK;
}

ns_status ns_greedy_argmax(const float* logits, int batch, int vocab, int32_t* out_ids, ns_stream_t stream) {
  if (!logits || !out_ids || batch < 1 || vocab < 1) return fail(NS_ERR_INVALID_ARG, "argmax arguments");
  NS_CUDA(launch_argmax(logits, batch, vocab, out_ids, reinterpret_cast<cudaStream_t>(stream)));
  return NS_OK;
}

}  // extern "C"

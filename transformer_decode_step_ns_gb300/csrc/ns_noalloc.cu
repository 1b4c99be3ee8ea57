// ns_attn_decode_noalloc: the paged decode-attention call for callers that cannot allocate
// device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- an allocator or memory-pool
// callback, a plugin whose host process owns every device allocation and forbids hidden ones,
// or a process that must not grow its device footprint after start-up.  ns_attn_decode grows
// a library-owned scratch buffer with cudaMalloc on first use; this variant instead uses a
// fixed buffer that is part of the loaded library image (a file-scope __device__ array), so a
// call never allocates or frees anything.
//
// The buffer holds the split-K partial results and the per-(row, kv head) arrival counters of
// the attention kernel.  Its size is fixed at build time (kNoAllocScratchBytes); requests that
// would need more are rejected.  Every call on a device shares the one buffer: two calls whose
// kernels overlap in time on that GPU (different streams, no ordering between them) race on it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "ns.h"
#include "ns_host.h"

namespace {

// 32 MiB of partials plus 64 Ki counters; every GPU that loads the library holds it until exit.
constexpr size_t kNoAllocPartialBytes = 32u << 20;
constexpr size_t kNoAllocCounters = 64u << 10;
constexpr size_t kNoAllocScratchBytes = kNoAllocPartialBytes + kNoAllocCounters * sizeof(int);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device (the symbol's host-side name is only a
// stand-in; it must be translated with that device current).  The address belongs to the
// context the module was loaded into, so each entry also records that context's unique id:
// after a device reset (or any teardown of the primary context) the module is loaded again,
// perhaps elsewhere, the id changes, and the next call looks the address up again.
struct ScratchSlot {
  unsigned long long ctx_id = 0;
  unsigned char* addr = nullptr;
};
std::mutex g_mu;
ScratchSlot g_slot[64];

// Unique id (cuCtxGetId) of the context current on this thread, or 0 when there is none or
// the driver entry points are unavailable (then the address is looked up on every call).
unsigned long long current_ctx_id() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (get_cur == nullptr || get_id == nullptr) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur(&c) != CUDA_SUCCESS || c == nullptr || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

ns_status scratch_address(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    ns::set_last_error("ns_attn_decode_noalloc: no usable current device");
    return NS_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchSlot& slot = g_slot[dev];
  const unsigned long long id = current_ctx_id();
  if (slot.addr == nullptr || id == 0 || id != slot.ctx_id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      ns::set_last_error((std::string("ns_attn_decode_noalloc: cudaGetSymbolAddress failed: ") +
                          cudaGetErrorString(e)).c_str());
      return NS_ERR_CUDA;
    }
    slot.addr = static_cast<unsigned char*>(p);
    slot.ctx_id = current_ctx_id();  // the lookup makes the primary context current if it was not
  }
  *out = slot.addr;
  return NS_OK;
}

}  // namespace

extern "C" ns_status ns_attn_decode_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                            const int32_t* block_tables, const int32_t* seq_lens,
                                            void* out, int batch, int n_q_heads, int n_kv_heads,
                                            int head_dim, int block_size, int max_blocks_per_seq,
                                            int num_blocks, float scale, int dtype, int* dev_err,
                                            ns_stream_t stream) {
  using namespace ns;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) {
    set_last_error("ns_attn_decode_noalloc: null argument");
    return NS_ERR_INVALID_ARG;
  }
  if (batch < 1 || batch > kMaxRows || n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads ||
      max_blocks_per_seq < 1 || num_blocks < 1 || !(scale > 0.f) ||
      (dtype != NS_F16 && dtype != NS_BF16)) {
    set_last_error("ns_attn_decode_noalloc: attention arguments");
    return NS_ERR_INVALID_ARG;
  }
  const int G = n_q_heads / n_kv_heads;
  if (!attn_supported(head_dim, G, block_size)) {
    set_last_error("ns_attn_decode_noalloc: attention shape not supported");
    return NS_ERR_UNSUPPORTED;
  }
  if (max_blocks_per_seq * block_size > 65536) {
    set_last_error("ns_attn_decode_noalloc: max_blocks_per_seq * block_size above 65536");
    return NS_ERR_UNSUPPORTED;
  }
  const int max_chunks = attn_max_chunks(max_blocks_per_seq * block_size);
  const size_t rows_heads = static_cast<size_t>(batch) * n_kv_heads;
  const size_t partial_bytes = rows_heads * attn_slot_floats(max_chunks, G, head_dim) * sizeof(float);
  if (partial_bytes > kNoAllocPartialBytes || rows_heads + 1 > kNoAllocCounters) {
    set_last_error(("ns_attn_decode_noalloc: request needs " + std::to_string(partial_bytes) +
                    " bytes of partials and " + std::to_string(rows_heads + 1) +
                    " counters; the fixed scratch holds " + std::to_string(kNoAllocPartialBytes) +
                    " bytes and " + std::to_string(kNoAllocCounters) +
                    " counters (reduce batch, kv heads or max_blocks_per_seq)").c_str());
    return NS_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(num_blocks) * n_kv_heads * block_size >= (1ll << 31)) {
    set_last_error("ns_attn_decode_noalloc: num_blocks * n_kv_heads * block_size must fit in int32");
    return NS_ERR_UNSUPPORTED;
  }
  unsigned char* base = nullptr;
  ns_status st = scratch_address(&base);
  if (st != NS_OK) return st;
  int* counters = reinterpret_cast<int*>(base + kNoAllocPartialBytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The counters (per (row, kv head), then the unit queue's) must start at zero; a call that
  // ended early could have left them dirty.
  cudaError_t e = cudaMemsetAsync(counters, 0, (rows_heads + 1) * sizeof(int), s);
  if (e != cudaSuccess) {
    set_last_error((std::string("ns_attn_decode_noalloc: ") + cudaGetErrorString(e)).c_str());
    return NS_ERR_CUDA;
  }
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
  ap.partials = reinterpret_cast<float*>(base);
  ap.counters = counters;
  ap.sched = reinterpret_cast<unsigned*>(counters + rows_heads);
  ap.err = dev_err;
  const long long units = static_cast<long long>(batch) * n_kv_heads * max_chunks;
  const int grid =
      static_cast<int>(std::min<long long>(attn_max_grid(dtype, head_dim, G, batch), units));
  // seq_lens are on the device: the queue variant whenever the rows could hold enough units
  e = launch_attn(ap, dtype, head_dim, G, grid, s, false,
                  units >= static_cast<long long>(kAttnQueueUnits) * grid);
  if (e != cudaSuccess) {
    set_last_error((std::string("ns_attn_decode_noalloc: launch: ") + cudaGetErrorString(e)).c_str());
    return NS_ERR_CUDA;
  }
  return NS_OK;
}

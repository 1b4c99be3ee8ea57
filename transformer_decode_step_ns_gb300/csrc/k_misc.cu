// Per-step token kernels: embedding gather fused with the RoPE table and the first RMSNorm's
// inputs, and the greedy argmax over the logits.
//
// "GPU waiting, not working" (nanoserve notes), change table: the RoPE cos/sin are built once
// per step (positions are shared by every layer) -- here in the same launch as the embedding
// gather, which also writes the first layer's RMSNorm input (x * gamma) and the per-128-column
// sums of squares that the QKV projection's epilogue turns into the norm scale.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ns_epi.cuh"
#include "ns_internal.h"
#include "ns_ptx.cuh"

namespace ns {

namespace {

template <typename T>
struct EV;
template <>
struct EV<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};
template <>
struct EV<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

}  // namespace

// grid = batch rows, block = 128 threads (one thread per column of each 128-column tile).  The
// row is read kEmbedTiles tiles at a time, all loads in flight before any result is used.
constexpr int kEmbedTiles = 16;

template <typename T>
__global__ void __launch_bounds__(128) embed_rope_kernel(const EmbedParams p) {
  __shared__ float warp_sums[kEmbedTiles][4];
  const int row = p.row0 + blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Token ids and positions are step metadata, complete before the step: read them early.
  int tok = (p.rows_valid != nullptr && row >= *p.rows_valid) ? 0 : p.token_ids[row];
  // -(r + 1): the token sampled at row r of the previous step, in the device token source (its
  // writer, the previous step's argmax, precedes this kernel without a programmatic edge)
  if (tok < 0 && p.tok_src != nullptr) tok = p.tok_src[-tok - 1];
  const int pos = p.positions[row];
  if (tid == 0) griddep_launch_dependents();
  griddep_wait();  // the residual/xn rows may still be read by the previous step's tail
  if (tok < 0 || tok >= p.vocab) {
    if (tid == 0) atomicCAS(p.err, 0, NS_DEV_BAD_TOKEN);
    tok = 0;
  }
  const T* e = reinterpret_cast<const T*>(p.embed) + static_cast<size_t>(tok) * p.hidden;
  T* xn = reinterpret_cast<T*>(p.xn) + static_cast<size_t>(row) * p.hidden;
  float* resid = p.resid + static_cast<size_t>(row) * p.hidden;
  const int n_tiles = p.hidden / 128;
  for (int t0 = 0; t0 < n_tiles; t0 += kEmbedTiles) {
    float v[kEmbedTiles], g[kEmbedTiles];
#pragma unroll
    for (int u = 0; u < kEmbedTiles; ++u) {
      const int i = (t0 + u) * 128 + tid;
      v[u] = t0 + u < n_tiles ? EV<T>::to_f(e[i]) : 0.f;
      g[u] = t0 + u < n_tiles ? p.gamma[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kEmbedTiles; ++u) {
      if (t0 + u >= n_tiles) break;
      const int i = (t0 + u) * 128 + tid;
      resid[i] = v[u];
      xn[i] = EV<T>::from_f(v[u] * g[u]);
      float s = v[u] * v[u];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) warp_sums[u][warp] = s;
    }
    __syncthreads();
    if (tid < kEmbedTiles && t0 + tid < n_tiles) {
      const float* w = warp_sums[tid];
      p.sumsq[static_cast<size_t>(t0 + tid) * p.sumsq_ld + row] = (w[0] + w[1]) + (w[2] + w[3]);
    }
    __syncthreads();
  }
  // RoPE table for this row (fp64 angle, Cody-Waite reduction, fp32 sincosf)
  const int half = p.head_dim / 2;
  for (int i = tid; i < half; i += 128) {
    float sn, cs;
    rope_cos_sin(pos, p.inv_freq[i], &cs, &sn);
    p.rope_cos[static_cast<size_t>(row) * half + i] = cs;
    p.rope_sin[static_cast<size_t>(row) * half + i] = sn;
  }
  fence_proxy_async_global();  // xn is read through TMA by the next kernel
}

// Greedy argmax; ties go to the lowest index, NaN never wins (an all-NaN row gives 0).  A
// cluster of kArgmaxSplit CTAs takes one row, each CTA a contiguous slice; rank 0 combines the
// slices' results through distributed shared memory (the comparison is a total order, so the
// result does not depend on the split).
constexpr int kArgmaxSplit = 8;

__device__ __forceinline__ void argmax_merge(float& best, int& bi, float ov, int oi) {
  if (ov > best || (ov == best && oi < bi)) {
    best = ov;
    bi = oi;
  }
}

constexpr int kArgmaxThreads = 256;

__global__ void __launch_bounds__(kArgmaxThreads) argmax_kernel(const float* logits, int vocab,
                                                                int32_t* out) {
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ int si[kArgmaxThreads / 32];
  const int row = blockIdx.y;
  const int rank = static_cast<int>(cluster_ctarank());
  const float* r = logits + static_cast<size_t>(row) * vocab;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  if ((vocab & 3) == 0) {
    // rows start on 16 bytes: 16-byte loads over slices of whole float4s
    const int n4 = vocab >> 2;
    const int per4 = (n4 + kArgmaxSplit - 1) / kArgmaxSplit;
    const int lo4 = rank * per4, hi4 = min(n4, lo4 + per4);
    const float4* r4 = reinterpret_cast<const float4*>(r);
#pragma unroll 4
    for (int i = lo4 + static_cast<int>(threadIdx.x); i < hi4; i += blockDim.x) {
      const float4 v = __ldg(r4 + i);
      argmax_merge(best, bi, v.x, 4 * i);
      argmax_merge(best, bi, v.y, 4 * i + 1);
      argmax_merge(best, bi, v.z, 4 * i + 2);
      argmax_merge(best, bi, v.w, 4 * i + 3);
    }
  } else {
    const int per = (vocab + kArgmaxSplit - 1) / kArgmaxSplit;
    const int lo = rank * per, hi = min(vocab, lo + per);
#pragma unroll 4
    for (int i = lo + static_cast<int>(threadIdx.x); i < hi; i += blockDim.x)
      argmax_merge(best, bi, r[i], i);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    argmax_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sv[warp] = best;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    best = lane < nw ? sv[lane] : -INFINITY;
    bi = lane < nw ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      argmax_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
    if (lane == 0) {
      sv[0] = best;  // this slice's result, read by rank 0
      si[0] = bi;
    }
  }
  cluster_sync();
  if (rank == 0 && warp == 0) {
    best = -INFINITY;
    bi = 0x7fffffff;
    if (lane < kArgmaxSplit) {
      best = ld_shared_cluster_f32(map_shared_rank(smem_u32(&sv[0]), lane));
      bi = static_cast<int>(ld_shared_cluster_u32(map_shared_rank(smem_u32(&si[0]), lane)));
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1)
      argmax_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
    if (lane == 0) out[row] = bi == 0x7fffffff ? 0 : bi;
  }
  cluster_sync();  // every slice stays resident until rank 0 has read it
}

// KV offload and reload (NanoFlow, "Runtime details that keep the pipeline fed"): K/V travel to
// and from the host as contiguous rows, and only on the device are they scattered into (or
// gathered from) the fragmented pages.  A thread moves one 16-byte piece per grid stride: 8
// elements of one head of one token; consecutive threads take consecutive pieces of a row, so
// both sides are coalesced (a head's d elements are contiguous in a page).  The index
// arithmetic is 32-bit when the piece count allows.
template <typename I>
__global__ void __launch_bounds__(256) kv_copy_kernel(const KvCopyParams p) {
  const int kvd = p.n_kv_heads * p.head_dim;
  const I per_row = kvd / 4;  // 16-byte pieces of a (layer, token) row of 2 * kvd elements
  const I total = static_cast<I>(p.n_layers) * p.n * per_row;
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  for (I u = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; u < total; u += stride) {
    const I r = u / per_row;
    const int c = static_cast<int>(u - r * per_row) * 8;  // element within the row
    const I l = r / p.n, t = r - l * p.n;
    const int kv = c >= kvd ? 1 : 0, col = c - kv * kvd;
    const int kvh = col / p.head_dim, dim = col - kvh * p.head_dim;
    const long long slot = p.slots[t];
    if (slot < 0 || slot >= p.pool_slots) {
      if (dim == 0) atomicCAS(p.err, 0, NS_DEV_BAD_SLOT);
      continue;
    }
    const size_t page = ((static_cast<size_t>(slot / p.block_size) * p.n_kv_heads + kvh) * p.block_size +
                         static_cast<size_t>(slot % p.block_size)) * p.head_dim + dim;
    uint4* pool = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.pools) +
                                           p.pool_bytes * (2 * static_cast<size_t>(l) + kv) + page * 2);
    uint4* row = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.buf) +
                                          (static_cast<size_t>(r) * 2 * kvd + c) * 2);
    if (p.to_pool) *pool = *row;
    else *row = *pool;
  }
}

// ------------------------------------------------------------------------------ host side

cudaError_t launch_kv_copy(const KvCopyParams& p, int sms, cudaStream_t s) {
  const long long pieces = static_cast<long long>(p.n_layers) * p.n * (p.n_kv_heads * p.head_dim / 4);
  if (pieces <= 0) return cudaSuccess;
  const bool narrow = pieces + 2LL * 256 * 16 * sms < (1LL << 31);  // u + stride stays in int32
  // one wave of resident CTAs (grid-stride beyond), fewer when the copy is small; the
  // occupancy of each instantiation is queried once (thread-safe static initialisation)
  auto occupancy = [](auto kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    return n;
  };
  static const int per_sm_narrow = occupancy(kv_copy_kernel<int>);
  static const int per_sm_wide = occupancy(kv_copy_kernel<long long>);
  const int ps = narrow ? per_sm_narrow : per_sm_wide;
  const long long need = (pieces + 255) / 256;
  const long long wave = static_cast<long long>(ps) * sms;
  const int grid = static_cast<int>(need < wave ? need : wave);
  if (narrow) kv_copy_kernel<int><<<grid, 256, 0, s>>>(p);
  else kv_copy_kernel<long long><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_embed(const EmbedParams& p, int dtype, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.batch, 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (dtype == NS_BF16) return cudaLaunchKernelEx(&cfg, embed_rope_kernel<__nv_bfloat16>, p);
  return cudaLaunchKernelEx(&cfg, embed_rope_kernel<__half>, p);
}

cudaError_t launch_argmax(const float* logits, int batch, int vocab, int32_t* out,
                          cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kArgmaxSplit, batch, 1);
  cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kArgmaxSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, argmax_kernel, logits, vocab, out);
}

}  // namespace ns

// Paged grouped-query decode attention with fixed-chunk split-K and an in-kernel merge.
//
// "GPU waiting, not working" (nanoserve notes), change table: grouped-query attention must
// not materialise the G-times expanded copy of K and V, and a fused paged-attention kernel
// replaced about ten ops per layer.  "NanoFlow ..." ("Four resource classes"): decode
// attention is the memory-bound class, so the kernel is built to stream K/V at HBM speed:
//
// * Work unit = (request b, kv head g, chunk of 256 tokens).  The chunking depends only on
//   seq_len, so a row's result never depends on the rest of the batch (nano-batch identity).
// * Persistent CTAs walk units round-robin.  One producer thread streams each (block, kv head)
//   K tile and V tile (block_size x d contiguous, 4 KiB at d=128 bf16) with cp.async.bulk into
//   an mbarrier ring; the producer runs ahead across unit boundaries.
// * Consumers: each K/V tile is read once from shared memory for all G query heads of its
//   group (no expansion).  QK: TPT threads per token, q held in registers, shuffle reduction;
//   online softmax in the log2 domain; PV: threads own dim pairs, token slices merged at the
//   end of the unit.
// * Chunks of one (b, g) are merged by the last-arriving CTA (atomic counter, no spin) in
//   chunk order with the log-sum-exp rule, so the result is deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ns_internal.h"
#include "ns_ptx.cuh"

namespace ns {

namespace {

template <typename T>
struct AV;  // vector helpers for the storage type
template <>
struct AV<__half> {
  static __device__ __forceinline__ float2 to2(uint32_t u) {
    return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(u & 0xffffu))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(u >> 16))));
  }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
};
template <>
struct AV<__nv_bfloat16> {
  static __device__ __forceinline__ float2 to2(uint32_t u) {
    // bf16 is the upper half of an fp32: widening is a shift
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
};

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

}  // namespace

template <int D, int G>
struct AttnShape {
  static constexpr int BS = 16;
  static constexpr int TPT = (G * D / 64 > 8) ? 16 : 8;  // QK threads per token (q regs <= 64)
  static constexpr int DPT = D / TPT;                               // dims per QK thread
  static constexpr int NC = BS * TPT;                               // consumer threads
  static constexpr int NWC = NC / 32;
  static constexpr int NT = NC + 32;                                // + producer warp
  static constexpr int DP = D / 2;                                  // PV dim pairs
  static constexpr int TS = NC / DP;                                // PV token slices
  static constexpr int TPS = BS / TS;                               // tokens per slice
  static constexpr int TILE = BS * D * 2;                           // bytes per K or V tile
  static constexpr int NSTAGE = (D == 128) ? 8 : 16;
  static constexpr int CHUNK_BLOCKS = kAttnChunkTokens / BS;
  static_assert(NC % 32 == 0 && TS * DP == NC && BS % TS == 0, "thread mapping");
  static_assert(DPT % 8 == 0, "16-byte K loads");
  // shared memory layout (bytes, from a 128-byte aligned base)
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_BAR = OFF_RING + NSTAGE * 2 * TILE;
  static constexpr int OFF_S = OFF_BAR + 2 * NSTAGE * 8;
  static constexpr int OFF_P = OFF_S + G * BS * 4;
  static constexpr int OFF_ML = OFF_P + BS * 8 * 4;          // m[8], l[8], alpha[8]
  static constexpr int OFF_FLAG = OFF_ML + 3 * 8 * 4;         // abort, last, total
  static constexpr int OFF_RED = OFF_FLAG + 16;
  static constexpr int OFF_PRE = OFF_RED + TS * G * D * 4;    // prefix over rows [batch + 1]
  static size_t smem_bytes(int batch) {
    return 128 + OFF_PRE + static_cast<size_t>(batch + 1) * 4;
  }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(AttnShape<D, G>::NT)
    attn_decode_kernel(const AttnParams p) {
  using S = AttnShape<D, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* empty = full + S::NSTAGE;
  float* s_sc = reinterpret_cast<float*>(smem + S::OFF_S);    // [G][BS] scores (log2 domain)
  float* s_p = reinterpret_cast<float*>(smem + S::OFF_P);     // [BS][8] probabilities
  float* s_m = reinterpret_cast<float*>(smem + S::OFF_ML);
  float* s_l = s_m + 8;
  float* s_a = s_m + 16;
  int* abort_flag = reinterpret_cast<int*>(smem + S::OFF_FLAG);
  int* last_flag = abort_flag + 1;
  int* s_stop = abort_flag + 2;
  float* red = reinterpret_cast<float*>(smem + S::OFF_RED);   // [TS][G][D]
  int* pre = reinterpret_cast<int*>(smem + S::OFF_PRE);        // chunk prefix over rows

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.n_kv_heads;
  const int batch = p.batch;

  if (tid == 0) {
    for (int s = 0; s < S::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], S::NWC);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Chunk prefix over the rows (metadata is final before the step starts, so this overlaps the
  // previous kernel under programmatic dependent launch).
  {
    const int per = (batch + S::NT - 1) / S::NT;
    const int lo = tid * per, hi = min(batch, lo + per);
    int run = 0;
    for (int b = lo; b < hi; ++b) {
      const int L = p.seq_lens[p.row0 + b];
      const int ok = (L >= 1 && L <= p.mb * p.block_size);
      run += ok ? (L + kAttnChunkTokens - 1) / kAttnChunkTokens : 0;
    }
    // exclusive scan of per-thread totals through shared memory (reuses the red buffer)
    int* tot = reinterpret_cast<int*>(red);
    tot[tid] = run;
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int i = 0; i < S::NT; ++i) {
        const int v = tot[i];
        tot[i] = acc;
        acc += v;
      }
      pre[batch] = acc;
    }
    __syncthreads();
    int acc = tot[tid];
    for (int b = lo; b < hi; ++b) {
      pre[b] = acc;
      const int L = p.seq_lens[p.row0 + b];
      const int ok = (L >= 1 && L <= p.mb * p.block_size);
      if (!ok) set_err(p.err, NS_DEV_BAD_LENGTH);
      acc += ok ? (L + kAttnChunkTokens - 1) / kAttnChunkTokens : 0;
    }
    __syncthreads();
  }
  const int total = pre[batch] * Hkv;
  if (tid == 0) griddep_launch_dependents();
  griddep_wait();  // q and this step's K/V come from the previous kernel

  auto decode_unit = [&](int u, int& b, int& g, int& chunk, int& L) {
    const int cg = u / Hkv;
    g = u - cg * Hkv;
    int lo = 0, hi = batch - 1;  // largest b with pre[b] <= cg
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= cg) lo = mid; else hi = mid - 1;
    }
    b = lo;
    chunk = cg - pre[b];
    L = p.seq_lens[p.row0 + b];
  };

  const T* kpool = reinterpret_cast<const T*>(p.k_pool);
  const T* vpool = reinterpret_cast<const T*>(p.v_pool);

  if (warp == S::NWC) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < total && !stop; u += gridDim.x) {
        int b, g, chunk, L;
        decode_unit(u, b, g, chunk, L);
        const int blk0 = chunk * S::CHUNK_BLOCKS;
        const int t_end = min(L, (chunk + 1) * kAttnChunkTokens);
        const int nblk = (t_end - chunk * kAttnChunkTokens + S::BS - 1) / S::BS;
        const int* row_tab = p.block_tables + static_cast<size_t>(p.row0 + b) * p.mb;
        for (int i = 0; i < nblk; ++i, ++it) {
          const int s = it % S::NSTAGE;
          if (it >= S::NSTAGE) {
            if (!mbar_wait(&empty[s], static_cast<uint32_t>((it / S::NSTAGE) - 1) & 1u, abort_flag)) {
              *abort_flag = 1;
              set_err(p.err, NS_DEV_WAIT_TIMEOUT);
              stop = true;
              break;
            }
          }
          int blk = row_tab[blk0 + i];
          if (blk < 0 || blk >= p.num_blocks) {
            set_err(p.err, NS_DEV_BAD_BLOCK);
            blk = 0;  // keep the pipeline consistent; the row's output is flagged invalid
          }
          const size_t off = (static_cast<size_t>(blk) * Hkv + g) * S::BS * D;
          uint8_t* dst = smem + S::OFF_RING + static_cast<size_t>(s) * 2 * S::TILE;
          mbar_arrive_expect_tx(&full[s], 2 * S::TILE);
          bulk_g2s_hint(dst, kpool + off, S::TILE, &full[s], pol);
          bulk_g2s_hint(dst + S::TILE, vpool + off, S::TILE, &full[s], pol);
        }
      }
      // drain: let copies in flight land before exit
      __threadfence_block();
      const int first = max(0, it - S::NSTAGE);
      for (int i = first; i < it; ++i) {
        (void)mbar_wait(&full[i % S::NSTAGE], static_cast<uint32_t>(i / S::NSTAGE) & 1u,
                        nullptr);
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int ct = tid;                 // 0..NC-1
  const int qt = ct / S::TPT;         // QK token
  const int qp = ct % S::TPT;         // QK part
  const int ts = ct / S::DP;          // PV token slice
  const int dp = ct % S::DP;          // PV dim pair
  int it = 0;
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    int b, g, chunk, L;
    decode_unit(u, b, g, chunk, L);
    const int t_begin = chunk * kAttnChunkTokens;
    const int t_end = min(L, t_begin + kAttnChunkTokens);
    const int nblk = (t_end - t_begin + S::BS - 1) / S::BS;
    const int nchunks = (L + kAttnChunkTokens - 1) / kAttnChunkTokens;
    const size_t row = static_cast<size_t>(p.row0 + b);

    float qr[G][S::DPT];
    {
      const T* qsrc = reinterpret_cast<const T*>(p.q) + row * p.q_row_stride +
                      static_cast<size_t>(g) * G * D + qp * S::DPT;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
#pragma unroll
        for (int v = 0; v < S::DPT / 8; ++v) {
          const uint4 raw = *reinterpret_cast<const uint4*>(qsrc + gg * D + v * 8);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = AV<T>::to2(w[k]);
            qr[gg][v * 8 + 2 * k] = f.x * p.scale_log2;
            qr[gg][v * 8 + 2 * k + 1] = f.y * p.scale_log2;
          }
        }
      }
    }
    if (ct < G) {
      s_m[ct] = -INFINITY;
      s_l[ct] = 0.f;
    }
    float acc[G][2];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) acc[gg][0] = acc[gg][1] = 0.f;

    bool failed = false;
    for (int i = 0; i < nblk; ++i, ++it) {
      const int s = it % S::NSTAGE;
      const bool got = mbar_wait(&full[s], static_cast<uint32_t>(it / S::NSTAGE) & 1u, abort_flag);
      if (!got) {
        *abort_flag = 1;
        set_err(p.err, NS_DEV_WAIT_TIMEOUT);
      }
      const uint8_t* kt = smem + S::OFF_RING + static_cast<size_t>(s) * 2 * S::TILE;
      const uint8_t* vt = kt + S::TILE;
      const int tok_base = t_begin + i * S::BS;
      // ---- QK: scores for token qt of this block, all G heads
      {
        float kf[S::DPT];
        const T* krow = reinterpret_cast<const T*>(kt) + qt * D + qp * S::DPT;
#pragma unroll
        for (int v = 0; v < S::DPT / 8; ++v) {
          uint4 raw = make_uint4(0u, 0u, 0u, 0u);
          if (got) raw = *reinterpret_cast<const uint4*>(krow + v * 8);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = AV<T>::to2(w[k]);
            kf[v * 8 + 2 * k] = f.x;
            kf[v * 8 + 2 * k + 1] = f.y;
          }
        }
        const bool valid = tok_base + qt < t_end;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          float sdot = 0.f;
#pragma unroll
          for (int k = 0; k < S::DPT; ++k) sdot = fmaf(qr[gg][k], kf[k], sdot);
#pragma unroll
          for (int o = S::TPT / 2; o > 0; o >>= 1) sdot += __shfl_xor_sync(0xffffffffu, sdot, o);
          if (qp == 0) s_sc[gg * S::BS + qt] = valid ? sdot : -INFINITY;
        }
      }
      named_barrier_sync(1, S::NC);
      // ---- online softmax: thread (gg, t) for ct < 16 G; every consumer lane takes part in
      // the shuffles (16-lane groups), only active lanes write.
      {
        const bool act = ct < S::BS * G;
        const int gg = act ? ct / S::BS : 0, t = ct % S::BS;
        const float sc = act ? s_sc[gg * S::BS + t] : 0.f;
        float mx = sc;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_old = s_m[gg];
        const float m_new = fmaxf(m_old, mx);
        const float pr = exp2f(sc - m_new);
        float sum = pr;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (ct == 0) s_stop[0] = *abort_flag;
        if (act) {
          s_p[t * 8 + gg] = pr;
          if (t == 0) {
            const float a = exp2f(m_old - m_new);
            s_a[gg] = a;
            s_l[gg] = s_l[gg] * a + sum;
            s_m[gg] = m_new;
          }
        }
      }
      named_barrier_sync(1, S::NC);
      if (s_stop[0]) {
        failed = true;
        break;
      }
      // ---- PV: dim pair dp, tokens of slice ts
      {
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float a = s_a[gg];
          acc[gg][0] *= a;
          acc[gg][1] *= a;
        }
        const uint32_t* vw = reinterpret_cast<const uint32_t*>(vt);
#pragma unroll
        for (int tt = 0; tt < S::TPS; ++tt) {
          const int t = ts * S::TPS + tt;
          if (tok_base + t < t_end) {
            const float2 v = AV<T>::to2(vw[t * S::DP + dp]);
            const float* pp = s_p + t * 8;
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
              const float pr = pp[gg];
              acc[gg][0] = fmaf(pr, v.x, acc[gg][0]);
              acc[gg][1] = fmaf(pr, v.y, acc[gg][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (failed) break;

    // ---- merge token slices; write the output or this chunk's partial
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      red[(ts * G + gg) * D + 2 * dp] = acc[gg][0];
      red[(ts * G + gg) * D + 2 * dp + 1] = acc[gg][1];
    }
    named_barrier_sync(1, S::NC);
    T* out = reinterpret_cast<T*>(p.out);
    if (nchunks == 1) {
      for (int idx = ct; idx < G * D; idx += S::NC) {
        const int gg = idx / D, dd = idx - gg * D;
        float o = 0.f;
#pragma unroll
        for (int k = 0; k < S::TS; ++k) o += red[(k * G + gg) * D + dd];
        out[row * p.out_row_stride + static_cast<size_t>(g * G + gg) * D + dd] =
            AV<T>::from_f(o / s_l[gg]);
      }
    } else {
      float* part = p.partials +
                    ((row * Hkv + g) * static_cast<size_t>(p.max_chunks) + chunk) * G * (D + 2);
      for (int idx = ct; idx < G * D; idx += S::NC) {
        const int gg = idx / D, dd = idx - gg * D;
        float o = 0.f;
#pragma unroll
        for (int k = 0; k < S::TS; ++k) o += red[(k * G + gg) * D + dd];
        part[gg * (D + 2) + dd] = o;
      }
      if (ct < G) {
        part[ct * (D + 2) + D] = s_m[ct];
        part[ct * (D + 2) + D + 1] = s_l[ct];
      }
      __threadfence();
      named_barrier_sync(1, S::NC);
      if (ct == 0) {
        int* cnt = p.counters + row * Hkv + g;
        const int old = atomicAdd(cnt, 1);
        const int last = (old == nchunks - 1) ? 1 : 0;
        if (last) *cnt = 0;
        *last_flag = last;
      }
      named_barrier_sync(1, S::NC);
      if (*last_flag) {
        __threadfence();
        const float* p0 = p.partials + (row * Hkv + g) * static_cast<size_t>(p.max_chunks) * G * (D + 2);
        for (int idx = ct; idx < G * D; idx += S::NC) {
          const int gg = idx / D, dd = idx - gg * D;
          float mmax = -INFINITY;
          for (int c = 0; c < nchunks; ++c) {
            const float* pc = p0 + static_cast<size_t>(c) * G * (D + 2) + gg * (D + 2);
            mmax = fmaxf(mmax, __ldcg(pc + D));
          }
          float lsum = 0.f, o = 0.f;
          for (int c = 0; c < nchunks; ++c) {
            const float* pc = p0 + static_cast<size_t>(c) * G * (D + 2) + gg * (D + 2);
            const float w = exp2f(__ldcg(pc + D) - mmax);
            lsum = fmaf(__ldcg(pc + D + 1), w, lsum);
            o = fmaf(__ldcg(pc + dd), w, o);
          }
          out[row * p.out_row_stride + static_cast<size_t>(g * G + gg) * D + dd] =
              AV<T>::from_f(o / lsum);
        }
      }
    }
    named_barrier_sync(1, S::NC);  // red / s_m / s_l are reused by the next unit
  }
}

// ------------------------------------------------------------------------------ host side

namespace {

template <typename T, int D, int G>
cudaError_t launch_attn_t(const AttnParams& p, int grid, cudaStream_t s, bool pdl) {
  using S = AttnShape<D, G>;
  static int configured_mask = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 31 && !(configured_mask & (1 << dev))) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<T, D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured_mask |= 1 << dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(S::NT, 1, 1);
  cfg.dynamicSmemBytes = S::smem_bytes(p.batch);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<T, D, G>, p);
}

template <typename T, int D>
cudaError_t dispatch_g(const AttnParams& p, int group, int grid, cudaStream_t s, bool pdl) {
  switch (group) {
    case 1: return launch_attn_t<T, D, 1>(p, grid, s, pdl);
    case 2: return launch_attn_t<T, D, 2>(p, grid, s, pdl);
    case 4: return launch_attn_t<T, D, 4>(p, grid, s, pdl);
    case 7: return launch_attn_t<T, D, 7>(p, grid, s, pdl);
    case 8: return launch_attn_t<T, D, 8>(p, grid, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D, int G>
int max_grid_t(int batch) {
  using S = AttnShape<D, G>;
  int dev = 0, sms = 1, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncSetAttribute(attn_decode_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       227 * 1024);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_decode_kernel<T, D, G>, S::NT,
                                                    S::smem_bytes(batch)) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return sms * per_sm;
}

template <typename T, int D>
int max_grid_g(int group, int batch) {
  switch (group) {
    case 1: return max_grid_t<T, D, 1>(batch);
    case 2: return max_grid_t<T, D, 2>(batch);
    case 4: return max_grid_t<T, D, 4>(batch);
    case 7: return max_grid_t<T, D, 7>(batch);
    default: return max_grid_t<T, D, 8>(batch);
  }
}

}  // namespace

bool attn_supported(int head_dim, int group, int block_size) {
  if (block_size != 16) return false;
  if (head_dim != 64 && head_dim != 128) return false;
  return group == 1 || group == 2 || group == 4 || group == 7 || group == 8;
}

int attn_max_grid(int dtype, int head_dim, int group, int batch) {
  if (dtype == NS_BF16)
    return head_dim == 64 ? max_grid_g<__nv_bfloat16, 64>(group, batch)
                          : max_grid_g<__nv_bfloat16, 128>(group, batch);
  return head_dim == 64 ? max_grid_g<__half, 64>(group, batch) : max_grid_g<__half, 128>(group, batch);
}

cudaError_t launch_attn(const AttnParams& p, int dtype, int head_dim, int group, int grid,
                        cudaStream_t s, bool pdl) {
  if (grid < 1) grid = 1;
  if (dtype == NS_BF16) {
    return head_dim == 64 ? dispatch_g<__nv_bfloat16, 64>(p, group, grid, s, pdl)
                          : dispatch_g<__nv_bfloat16, 128>(p, group, grid, s, pdl);
  }
  return head_dim == 64 ? dispatch_g<__half, 64>(p, group, grid, s, pdl)
                        : dispatch_g<__half, 128>(p, group, grid, s, pdl);
}

}  // namespace ns

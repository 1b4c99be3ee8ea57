// Paged grouped-query decode attention: warp-independent units, TMA-staged K/V tiles,
// tensor-core (mma.sync m16n8k16) QK^T and PV, split-K over fixed chunks with an in-kernel merge.
//
// "GPU waiting, not working" (nanoserve notes), change table: grouped-query attention must not
// materialise the G-times expanded copy of K and V, and one fused paged-attention kernel
// replaces about ten ops per layer.  "NanoFlow ..." ("Four resource classes"): decode attention
// is the memory-bound class, so the kernel is built to stream K/V at HBM speed:
//
// * Work unit = (request b, kv head g, chunk).  A row of length L splits into chunks of
//   128 * ceil(L / 2048) tokens (at most 16 chunks); the chunking is a function of L alone, so a
//   row's result never depends on the rest of the batch.
// * Every warp walks its own units (round-robin over all warps of the grid) with a private ring
//   of TMA tensor copies: one 16 x d K tile and one V tile per cache block, 128-byte swizzled so
//   the ldmatrix reads below are bank-conflict free.  The warp refills a stage as soon as it has
//   consumed it and runs ahead across unit boundaries.  A unit's block ids are copied to shared
//   memory (cp.async) one unit ahead, and its q one unit ahead into registers, so the stream
//   never waits on a block-table or q read.
// * The G <= 8 query heads of the group form the rows of one 16-row mma.sync tile:
//     S^T[head][token]  = q[head][:] . K[token][:]          (A = q in registers, B = K tile)
//     O^T[dim][head]   += V^T[dim][token] . P^T[token][head] (A = V tile via ldmatrix.trans)
//   The accumulator layout of the first product is exactly the B-operand layout of the second,
//   so P never leaves registers.  Each K/V element is read once from shared memory for all G
//   heads: no expansion.  Online softmax in the log2 domain, per head, in registers.
// * Chunks of one (b, g) are merged by the last-arriving warp (atomic counter, no spin) in chunk
//   order with the log-sum-exp rule: deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ns_internal.h"
#include "ns_ptx.cuh"

namespace ns {

namespace {

template <typename T>
struct MV;
template <>
struct MV<__half> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};
template <>
struct MV<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

}  // namespace

template <int D, int G>
struct AttnShape {
  static constexpr int NW = 4;                 // independent warps per CTA
  static constexpr int NT = NW * 32;
  static constexpr int BS = 16;                // tokens per cache block
  static constexpr int NH = D / 64;            // 128-byte column halves of a tile
  static constexpr int TILE = BS * D * 2;      // bytes of one K or V tile
  static constexpr int STAGE = 2 * TILE;
  static constexpr int NST = (D == 128) ? 3 : 6;
  static constexpr int KS = D / 16;            // QK k-steps = PV m-tiles
  static constexpr int RING = NST * STAGE;     // bytes per warp
  static constexpr int OFF_BAR = NW * RING;
  static constexpr int OFF_FLAG = OFF_BAR + NW * NST * 8;
  static constexpr int OFF_IDS = OFF_FLAG + 16;  // per warp, 2 slots x ids_cap block ids
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(G >= 1 && G <= 8, "group");
  // then chunk prefix [batch + 1], lengths [batch], scan scratch [NT]
  static size_t smem_bytes(int batch, int ids_cap) {
    return 1024 + OFF_IDS + static_cast<size_t>(NW) * 2 * ids_cap * 4 +
           static_cast<size_t>(2 * batch + 1 + NT) * 4;
  }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(AttnShape<D, G>::NT, 2)
    attn_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  using S = AttnShape<D, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* abort_flag = reinterpret_cast<int*>(smem + S::OFF_FLAG);
  int* ids_all = reinterpret_cast<int*>(smem + S::OFF_IDS);  // [NW][2][ids_cap]
  int* pre = ids_all + S::NW * 2 * p.ids_cap;                 // chunk prefix over rows [batch + 1]
  int* lens = pre + p.batch + 1;                              // validated seq_lens [batch]
  int* tot = lens + p.batch;                                  // per-thread scan scratch [NT]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.n_kv_heads, batch = p.batch;
  uint8_t* ring = smem + warp * S::RING;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR) + warp * S::NST;

  if (lane == 0) {
    for (int s = 0; s < S::NST; ++s) mbar_init(&full[s], 1);
  }
  if (tid == 0) *abort_flag = 0;
  // Chunk prefix over the rows.  seq_lens are step metadata, final before the step starts, so
  // under programmatic dependent launch this overlaps the previous kernel.
  {
    const int per = (batch + S::NT - 1) / S::NT;
    const int lo = tid * per, hi = min(batch, lo + per);
    int run = 0;
    for (int b = lo; b < hi; ++b) {
      const int L = p.seq_lens[p.row0 + b];
      const bool ok = L >= 1 && L <= p.mb * p.block_size;
      if (!ok) set_err(p.err, NS_DEV_BAD_LENGTH);
      lens[b] = ok ? L : 0;
      run += ok ? attn_num_chunks(L) : 0;
    }
    tot[tid] = run;
    fence_mbar_init();
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
      acc += attn_num_chunks(lens[b]);
    }
    __syncthreads();
  }
  const int total = pre[batch] * Hkv;
  if (tid == 0) griddep_launch_dependents();
  griddep_wait();  // q and this step's K/V come from the previous kernel

  struct Unit {
    int b, g, chunk, L, t0, t1, nblk, nchunks;
  };
  auto decode = [&](int u) {
    Unit x;
    const int cg = u / Hkv;
    x.g = u - cg * Hkv;
    int lo = 0, hi = batch - 1;  // largest b with pre[b] <= cg
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= cg) lo = mid; else hi = mid - 1;
    }
    x.b = lo;
    x.chunk = cg - pre[lo];
    x.L = lens[lo];
    const int ct = attn_chunk_tokens(x.L);
    x.t0 = x.chunk * ct;
    x.t1 = min(x.L, x.t0 + ct);
    x.nblk = (x.t1 - x.t0 + S::BS - 1) / S::BS;
    x.nchunks = attn_num_chunks(x.L);
    return x;
  };

  const int gw = blockIdx.x * S::NW + warp, TW = gridDim.x * S::NW;

  // ---- producer cursor (warp-uniform): the warp's stream of (unit, block) in consumption order
  int* ids = ids_all + warp * 2 * p.ids_cap;
  auto prefetch_ids = [&](int unit, int slot) {
    if (unit < total) {
      const Unit x = decode(unit);
      const int* src = p.block_tables + static_cast<size_t>(p.row0 + x.b) * p.mb + x.t0 / S::BS;
      for (int j = lane; j < x.nblk; j += 32) cp_async_4(ids + slot * p.ids_cap + j, src + j);
    }
    cp_async_commit();
  };
  int pu = gw, pi = 0, ps = 0, issued = 0;
  Unit pun{};
  auto enter = [&]() {  // the producer starts unit pu (slot ps): its ids were prefetched
    cp_async_wait_all();
    __syncwarp();
    if (pu < total) pun = decode(pu);
    prefetch_ids(pu + TW, ps ^ 1);
  };
  prefetch_ids(pu, 0);
  enter();
  auto issue = [&](int stage) {  // warp-collective; lane 0 issues the copies
    if (pu >= total) return;
    int blk = ids[ps * p.ids_cap + pi];
    if (blk < 0 || blk >= p.num_blocks) {
      if (lane == 0) set_err(p.err, NS_DEV_BAD_BLOCK);
      blk = 0;  // keep the pipeline consistent; the error word flags the result
    }
    if (lane == 0) {
      uint8_t* dst = ring + stage * S::STAGE;
      const int y = (blk * Hkv + pun.g) * S::BS;
      mbar_arrive_expect_tx(&full[stage], S::STAGE);
#pragma unroll
      for (int h = 0; h < S::NH; ++h) {
        tma_load_2d(dst + h * 2048, &kmap, &full[stage], h * 64, y);
        tma_load_2d(dst + S::TILE + h * 2048, &vmap, &full[stage], h * 64, y);
      }
    }
    ++issued;
    if (++pi >= pun.nblk) {
      pi = 0;
      pu += TW;
      ps ^= 1;
      enter();
    }
  };
  for (int s = 0; s < S::NST; ++s) issue(s);

  const int gq = lane >> 2, tq = lane & 3;
  // ldmatrix lane address: token row and 16-byte chunk offset within the 4 matrices
  const int lm_tok = (lane & 7) + ((lane >> 4) << 3);
  const int lm_chunk = (lane >> 3) & 1;
  T* out = reinterpret_cast<T*>(p.out);

  // q of the group as the A operand (rows = heads, G of 16 used; k = dims), loaded one unit
  // ahead so the loads overlap the previous unit's blocks.
  uint32_t qn[S::KS][2];
  auto load_q = [&](int unit) {
    if (unit >= total || gq >= G) {
#pragma unroll
      for (int ks = 0; ks < S::KS; ++ks) qn[ks][0] = qn[ks][1] = 0u;
      return;
    }
    const Unit x = decode(unit);
    const T* qrow = reinterpret_cast<const T*>(p.q) + static_cast<size_t>(p.row0 + x.b) * p.q_row_stride +
                    static_cast<size_t>(x.g * G + gq) * D;
#pragma unroll
    for (int ks = 0; ks < S::KS; ++ks) {
      qn[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tq);
      qn[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tq);
    }
  };
  load_q(gw);

  int ci = 0;
  bool failed = false;
  for (int u = gw; u < total && !failed; u += TW) {
    const Unit x = decode(u);
    const size_t row = static_cast<size_t>(p.row0 + x.b);
    uint32_t qa[S::KS][2];
#pragma unroll
    for (int ks = 0; ks < S::KS; ++ks) {
      qa[ks][0] = qn[ks][0];
      qa[ks][1] = qn[ks][1];
    }
    load_q(u + TW);
    float m_run = -INFINITY, l_run = 0.f;
    float acc[S::KS][4];
#pragma unroll
    for (int mt = 0; mt < S::KS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

    for (int i = 0; i < x.nblk; ++i, ++ci) {
      const int s = ci % S::NST;
      if (!mbar_wait(&full[s], static_cast<uint32_t>(ci / S::NST) & 1u, abort_flag)) {
        *abort_flag = 1;
        set_err(p.err, NS_DEV_WAIT_TIMEOUT);
        failed = true;
      }
      failed = __any_sync(0xffffffffu, failed);
      if (failed) break;
      const uint8_t* kt = ring + s * S::STAGE;
      const uint8_t* vt = kt + S::TILE;
      const int n_valid = min(S::BS, x.t1 - (x.t0 + i * S::BS));
      const bool zeroed = n_valid < S::BS;
      if (zeroed) {
        // stale slots past seq_len: zero their V rows so 0 * (anything) stays 0
        uint4* v4 = reinterpret_cast<uint4*>(const_cast<uint8_t*>(vt));
        for (int c = lane; c < S::BS * S::NH * 8; c += 32) {
          const int h = c / (S::BS * 8), r = (c / 8) % S::BS;
          if (r >= n_valid) v4[h * 128 + r * 8 + (c & 7)] = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
      const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
      // ---- S^T = q K^T: two n-tiles of 8 tokens; even / odd k-steps accumulate separately,
      // which halves the dependent MMA chain
      float sacc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < S::KS; ++ks) {
        const int chunk16 = 2 * ks + lm_chunk;           // 16-byte chunk = 8 dims
        const int h = chunk16 >> 3, cc = chunk16 & 7;
        const uint32_t addr = kbase + h * 2048 + lm_tok * 128 + ((cc ^ (lm_tok & 7)) << 4);
        uint32_t kb[4];
        ldsm_x4(addr, kb);
        const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
        MV<T>::mma(sacc[(ks & 1) * 2 + 0], a, kb[0], kb[1]);
        MV<T>::mma(sacc[(ks & 1) * 2 + 1], a, kb[2], kb[3]);
      }
      // ---- online softmax for head gq over tokens 2tq, 2tq+1, 8+2tq, 9+2tq
      float sc[4] = {sacc[0][0] + sacc[2][0], sacc[0][1] + sacc[2][1], sacc[1][0] + sacc[3][0],
                     sacc[1][1] + sacc[3][1]};
      const int tk[4] = {2 * tq, 2 * tq + 1, 8 + 2 * tq, 9 + 2 * tq};
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sc[k] = tk[k] < n_valid ? sc[k] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, sc[k]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = exp2f(m_run - m_new);
      float pr[4], psum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pr[k] = exp2f(sc[k] - m_new);
        psum += pr[k];
      }
      psum += __shfl_xor_sync(0xffffffffu, psum, 1);
      psum += __shfl_xor_sync(0xffffffffu, psum, 2);
      l_run = l_run * alpha + psum;
      m_run = m_new;
      // ---- O^T += V^T P^T  (P^T in the B-operand layout straight from the S^T accumulator)
      const uint32_t pb0 = MV<T>::pack(pr[0], pr[1]);
      const uint32_t pb1 = MV<T>::pack(pr[2], pr[3]);
      const float a_e = __shfl_sync(0xffffffffu, alpha, 8 * tq);      // head 2tq
      const float a_o = __shfl_sync(0xffffffffu, alpha, 8 * tq + 4);  // head 2tq + 1
#pragma unroll
      for (int mt = 0; mt < S::KS; ++mt) {
        acc[mt][0] *= a_e;
        acc[mt][1] *= a_o;
        acc[mt][2] *= a_e;
        acc[mt][3] *= a_o;
        const int chunk16 = 2 * mt + lm_chunk;
        const int h = chunk16 >> 3, cc = chunk16 & 7;
        const uint32_t addr = vbase + h * 2048 + lm_tok * 128 + ((cc ^ (lm_tok & 7)) << 4);
        uint32_t va[4];
        ldsm_x4_t(addr, va);
        MV<T>::mma(acc[mt], va, pb0, pb1);
      }
      // ---- the stage is consumed: refill it with the next block of this warp's stream
      __syncwarp();
      // generic-proxy zero writes must be ordered before the TMA overwrite of this stage
      if (zeroed && lane == 0) fence_proxy_async_smem();
      issue(s);
    }
    if (failed) break;

    // ---- unit result: heads 2tq and 2tq + 1 of this lane's accumulator columns
    const float l_e = __shfl_sync(0xffffffffu, l_run, 8 * tq);
    const float l_o = __shfl_sync(0xffffffffu, l_run, 8 * tq + 4);
    const int h_e = 2 * tq, h_o = 2 * tq + 1;
    if (x.nchunks == 1) {
      T* orow = out + row * p.out_row_stride + static_cast<size_t>(x.g) * G * D;
#pragma unroll
      for (int mt = 0; mt < S::KS; ++mt) {
        const int d0 = mt * 16 + gq;
        if (h_e < G) {
          orow[h_e * D + d0] = MV<T>::from_f(acc[mt][0] / l_e);
          orow[h_e * D + d0 + 8] = MV<T>::from_f(acc[mt][2] / l_e);
        }
        if (h_o < G) {
          orow[h_o * D + d0] = MV<T>::from_f(acc[mt][1] / l_o);
          orow[h_o * D + d0 + 8] = MV<T>::from_f(acc[mt][3] / l_o);
        }
      }
    } else {
      const size_t slot0 = (row * Hkv + x.g) * static_cast<size_t>(p.max_chunks);
      float* part = p.partials + (slot0 + x.chunk) * G * (D + 2);
#pragma unroll
      for (int mt = 0; mt < S::KS; ++mt) {
        const int d0 = mt * 16 + gq;
        if (h_e < G) {
          part[h_e * (D + 2) + d0] = acc[mt][0];
          part[h_e * (D + 2) + d0 + 8] = acc[mt][2];
        }
        if (h_o < G) {
          part[h_o * (D + 2) + d0] = acc[mt][1];
          part[h_o * (D + 2) + d0 + 8] = acc[mt][3];
        }
      }
      if (tq == 0 && gq < G) {
        part[gq * (D + 2) + D] = m_run;
        part[gq * (D + 2) + D + 1] = l_run;
      }
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        int* cnt = p.counters + row * Hkv + x.g;
        last = (atomicAdd(cnt, 1) == x.nchunks - 1) ? 1 : 0;
        if (last) *cnt = 0;  // ready for the next launch
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        const float* p0 = p.partials + slot0 * G * (D + 2);
        T* orow = out + row * p.out_row_stride + static_cast<size_t>(x.g) * G * D;
        for (int hh = 0; hh < G; ++hh) {
          // lane c < nchunks holds chunk c's (m, l); weights 2^(m_c - M), summed in chunk order
          float mc = -INFINITY, lc = 0.f;
          if (lane < x.nchunks) {
            mc = __ldcg(p0 + (static_cast<size_t>(lane) * G + hh) * (D + 2) + D);
            lc = __ldcg(p0 + (static_cast<size_t>(lane) * G + hh) * (D + 2) + D + 1);
          }
          float M = mc;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
          const float w = lane < x.nchunks ? exp2f(mc - M) : 0.f;
          float Lsum = 0.f;
          for (int c = 0; c < x.nchunks; ++c)
            Lsum = fmaf(__shfl_sync(0xffffffffu, lc, c), __shfl_sync(0xffffffffu, w, c), Lsum);
          for (int dd = lane; dd < D; dd += 32) {
            float o = 0.f;
            for (int c = 0; c < x.nchunks; ++c) {
              const float wc = __shfl_sync(0xffffffffu, w, c);
              o = fmaf(__ldcg(p0 + (static_cast<size_t>(c) * G + hh) * (D + 2) + dd), wc, o);
            }
            orow[hh * D + dd] = MV<T>::from_f(o / Lsum);
          }
        }
      }
    }
  }
  // On the normal path every issued copy was consumed.  After a timed-out wait, copies this
  // warp issued but did not consume must land before the CTA releases its shared memory.
  __syncwarp();
  cp_async_wait_all();
  if (failed && lane == 0) {
    for (int c = ci; c < issued; ++c) {
      (void)mbar_wait(&full[c % S::NST], static_cast<uint32_t>(c / S::NST) & 1u, nullptr);
    }
  }
}

// ------------------------------------------------------------------------------ host side

namespace {

template <typename T, int D, int G>
cudaError_t launch_attn_t(const AttnParams& p, const CUtensorMap* km, const CUtensorMap* vm,
                          int grid, cudaStream_t s, bool pdl) {
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
  cfg.dynamicSmemBytes = S::smem_bytes(p.batch, p.ids_cap);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<T, D, G>, *km, *vm, p);
}

template <typename T, int D>
cudaError_t dispatch_g(const AttnParams& p, const CUtensorMap* km, const CUtensorMap* vm,
                       int group, int grid, cudaStream_t s, bool pdl) {
  switch (group) {
    case 1: return launch_attn_t<T, D, 1>(p, km, vm, grid, s, pdl);
    case 2: return launch_attn_t<T, D, 2>(p, km, vm, grid, s, pdl);
    case 4: return launch_attn_t<T, D, 4>(p, km, vm, grid, s, pdl);
    case 7: return launch_attn_t<T, D, 7>(p, km, vm, grid, s, pdl);
    case 8: return launch_attn_t<T, D, 8>(p, km, vm, grid, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D, int G>
int max_grid_t(int batch, int ids_cap) {
  using S = AttnShape<D, G>;
  int dev = 0, sms = 1, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncSetAttribute(attn_decode_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       227 * 1024);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_decode_kernel<T, D, G>, S::NT,
                                                    S::smem_bytes(batch, ids_cap)) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return sms * per_sm;
}

template <typename T, int D>
int max_grid_g(int group, int batch, int ids_cap) {
  switch (group) {
    case 1: return max_grid_t<T, D, 1>(batch, ids_cap);
    case 2: return max_grid_t<T, D, 2>(batch, ids_cap);
    case 4: return max_grid_t<T, D, 4>(batch, ids_cap);
    case 7: return max_grid_t<T, D, 7>(batch, ids_cap);
    default: return max_grid_t<T, D, 8>(batch, ids_cap);
  }
}

}  // namespace

bool attn_supported(int head_dim, int group, int block_size) {
  if (block_size != 16) return false;
  if (head_dim != 64 && head_dim != 128) return false;
  return group == 1 || group == 2 || group == 4 || group == 7 || group == 8;
}

int attn_max_grid(int dtype, int head_dim, int group, int batch, int ids_cap) {
  if (dtype == NS_BF16)
    return head_dim == 64 ? max_grid_g<__nv_bfloat16, 64>(group, batch, ids_cap)
                          : max_grid_g<__nv_bfloat16, 128>(group, batch, ids_cap);
  return head_dim == 64 ? max_grid_g<__half, 64>(group, batch, ids_cap)
                        : max_grid_g<__half, 128>(group, batch, ids_cap);
}

cudaError_t launch_attn(const AttnParams& p, const CUtensorMap* kmap, const CUtensorMap* vmap,
                        int dtype, int head_dim, int group, int grid, cudaStream_t s, bool pdl) {
  if (grid < 1) grid = 1;
  if (dtype == NS_BF16) {
    return head_dim == 64 ? dispatch_g<__nv_bfloat16, 64>(p, kmap, vmap, group, grid, s, pdl)
                          : dispatch_g<__nv_bfloat16, 128>(p, kmap, vmap, group, grid, s, pdl);
  }
  return head_dim == 64 ? dispatch_g<__half, 64>(p, kmap, vmap, group, grid, s, pdl)
                        : dispatch_g<__half, 128>(p, kmap, vmap, group, grid, s, pdl);
}

}  // namespace ns

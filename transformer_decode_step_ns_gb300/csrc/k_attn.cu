// Paged grouped-query decode attention: warp-independent units, cp.async-staged K/V tiles,
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
//   of stages; each stage holds one 16 x d K tile and one V tile of a cache block, copied with
//   16-byte cp.async by all 32 lanes (each tile is one contiguous run, so every warp request is a
//   coalesced 512-byte read) into an XOR-swizzled layout that keeps the ldmatrix reads below
//   bank-conflict free.  Small per-block copies go through the load/store path rather than the
//   TMA engine, whose per-request cost limits throughput at 2-4 KiB tiles.  The warp refills a
//   stage as soon as it has consumed it and runs ahead across unit boundaries; q of the next unit
//   is loaded one unit ahead into registers.
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

// 16-byte global -> shared copy bypassing L1, with an L2 eviction-priority hint.
__device__ __forceinline__ void cp_async_16(uint32_t smem_dst, const void* gsrc, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_dst),
               "l"(gsrc), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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
  static constexpr int CPL = 2 * BS * D / 8 / 32;  // 16-byte copies per lane per stage
  static constexpr int OFF_MRG = NW * RING;    // per warp, [2][8][16] floats of merge scratch
  static constexpr int OFF_IDS = OFF_MRG + NW * 256 * 4;  // per warp, ids of the producer unit
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(G >= 1 && G <= 8, "group");
  // then chunk prefix [batch + 1], lengths [batch], scan scratch [NT]
  static size_t smem_bytes(int batch, int ids_cap) {
    return 1024 + OFF_IDS + static_cast<size_t>(NW) * ids_cap * 4 +
           static_cast<size_t>(2 * batch + 1 + NT) * 4;
  }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(AttnShape<D, G>::NT, 2) attn_decode_kernel(const AttnParams p) {
  using S = AttnShape<D, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* merge_all = reinterpret_cast<float*>(smem + S::OFF_MRG);  // [NW][2][8][16]
  int* ids_all = reinterpret_cast<int*>(smem + S::OFF_IDS);  // [NW][ids_cap]
  int* pre = ids_all + S::NW * p.ids_cap;                     // chunk prefix over rows [batch + 1]
  int* lens = pre + p.batch + 1;                              // validated seq_lens [batch]
  int* tot = lens + p.batch;                                  // per-thread scan scratch [NT]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.n_kv_heads, batch = p.batch;
  uint8_t* ring = smem + warp * S::RING;
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

  // ---- producer cursor (warp-uniform): the warp's stream of (unit, block) in consumption
  // order.  The block ids of the next unit are loaded into registers (lane j holds ids j,
  // j + 32, ...) when the producer enters the current one, and stored to shared memory when it
  // reaches the next, so the stream never waits on a block-table read.  Every stage is one
  // cp.async group, so "oldest stage landed" is wait_group(NST - 1).
  int* ids = ids_all + warp * p.ids_cap;
  const uint64_t pol = policy_evict_first();  // K/V are streamed once
  const T* kpool = reinterpret_cast<const T*>(p.k_pool);
  const T* vpool = reinterpret_cast<const T*>(p.v_pool);
  int pu = gw, pi = 0;
  Unit pun{}, nun{};
  int nid[kAttnIdRegs];
  auto load_ids = [&](int unit) {  // registers <- block ids of `unit` (non-blocking loads)
    nun = decode(unit);
    const int* src = p.block_tables + static_cast<size_t>(p.row0 + nun.b) * p.mb + nun.t0 / S::BS;
#pragma unroll
    for (int k = 0; k < kAttnIdRegs; ++k) {
      const int j = lane + 32 * k;
      nid[k] = j < nun.nblk ? src[j] : 0;
    }
  };
  auto enter = [&]() {  // the producer starts unit pu; its ids are in the registers
    __syncwarp();
    if (pu < total) {
      pun = nun;
#pragma unroll
      for (int k = 0; k < kAttnIdRegs; ++k) {
        const int j = lane + 32 * k;
        if (j < pun.nblk) {
          int blk = nid[k];
          if (blk < 0 || blk >= p.num_blocks) {
            set_err(p.err, NS_DEV_BAD_BLOCK);
            blk = 0;  // keep the pipeline consistent; the error word flags the result
          }
          ids[j] = blk;
        }
      }
      if (pu + TW < total) load_ids(pu + TW);
    }
    __syncwarp();
  };
  if (pu < total) load_ids(pu);
  enter();
  auto issue = [&](int stage) {  // warp-collective: one cp.async group per call
    if (pu < total) {
      const size_t tile_off = (static_cast<size_t>(ids[pi]) * Hkv + pun.g) * S::BS * D;
      const uint8_t* ksrc = reinterpret_cast<const uint8_t*>(kpool + tile_off);
      const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(vpool + tile_off);
      const uint32_t dst = smem_u32(ring + stage * S::STAGE);
#pragma unroll
      for (int k = 0; k < S::CPL; ++k) {
        const int c = lane + 32 * k;                  // chunk over [K | V] x 16 rows x D/8
        const int kv = c / (S::BS * D / 8);           // 0 = K, 1 = V
        const int ci16 = c - kv * (S::BS * D / 8);
        const int t = ci16 / (D / 8), c16 = ci16 % (D / 8);
        const int h = c16 >> 3, cc = c16 & 7;
        const uint32_t d_off = kv * S::TILE + h * 2048 + t * 128 + ((cc ^ (t & 7)) << 4);
        cp_async_16(dst + d_off, (kv ? vsrc : ksrc) + ci16 * 16, pol);
      }
      if (++pi >= pun.nblk) {
        pi = 0;
        pu += TW;
        enter();
      }
    }
    cp_async_commit();
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
  for (int u = gw; u < total; u += TW) {
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
      cp_async_wait_group<S::NST - 1>();  // this lane's copies of the oldest stage landed
      __syncwarp();                       // ... and every other lane's
      const uint8_t* kt = ring + s * S::STAGE;
      const uint8_t* vt = kt + S::TILE;
      const int n_valid = min(S::BS, x.t1 - (x.t0 + i * S::BS));
      if (n_valid < S::BS) {
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
      issue(s);
    }

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
      // partial slot of (row, kv head): acc [max_chunks][G][D], then (m, l) [max_chunks][G][2]
      float* pacc = p.partials + (row * Hkv + x.g) * attn_slot_floats(p.max_chunks, G, D);
      float* pml = pacc + static_cast<size_t>(p.max_chunks) * G * D;
      float* part = pacc + static_cast<size_t>(x.chunk) * G * D;
#pragma unroll
      for (int mt = 0; mt < S::KS; ++mt) {
        const int d0 = mt * 16 + gq;
        if (h_e < G) {
          part[h_e * D + d0] = acc[mt][0];
          part[h_e * D + d0 + 8] = acc[mt][2];
        }
        if (h_o < G) {
          part[h_o * D + d0] = acc[mt][1];
          part[h_o * D + d0 + 8] = acc[mt][3];
        }
      }
      if (tq == 0 && gq < G)
        reinterpret_cast<float2*>(pml)[x.chunk * G + gq] = make_float2(m_run, l_run);
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
        // Merge the chunks: weight_c = 2^(m_c - M) / sum_c' l_c' 2^(m_c' - M), summed in chunk
        // order.  One round trip for every (m, l), then one per head for the accumulators.
        __threadfence();
        float* mw = merge_all + warp * 256;  // [2][8 heads][16 chunks]
        const int nml = x.nchunks * G;       // <= 128
        float2 ml[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = lane + 32 * k;
          ml[k] = i < nml ? __ldcg(reinterpret_cast<const float2*>(pml) + i) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = lane + 32 * k;
          if (i < nml) {
            const int c = i / G, hh = i - c * G;
            mw[hh * 16 + c] = ml[k].x;
            mw[128 + hh * 16 + c] = ml[k].y;
          }
        }
        __syncwarp();
        if (lane < G) {
          float M = -INFINITY;
          for (int c = 0; c < x.nchunks; ++c) M = fmaxf(M, mw[lane * 16 + c]);
          float Lsum = 0.f;
          for (int c = 0; c < x.nchunks; ++c) Lsum = fmaf(mw[128 + lane * 16 + c], exp2f(mw[lane * 16 + c] - M), Lsum);
          const float inv = 1.f / Lsum;
          for (int c = 0; c < x.nchunks; ++c) mw[lane * 16 + c] = exp2f(mw[lane * 16 + c] - M) * inv;
        }
        __syncwarp();
        T* orow = out + row * p.out_row_stride + static_cast<size_t>(x.g) * G * D;
        constexpr int VW = D / 32;  // dims per lane: 4 (d = 128) or 2 (d = 64)
        for (int hh = 0; hh < G; ++hh) {
          float o[VW];
#pragma unroll
          for (int e = 0; e < VW; ++e) o[e] = 0.f;
          for (int cb = 0; cb < x.nchunks; cb += 8) {  // 8 chunks' loads in flight at a time
            float v[8][VW];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              if (cb + c < x.nchunks) {
                const float* src = pacc + (static_cast<size_t>(cb + c) * G + hh) * D + VW * lane;
                if constexpr (VW == 4) {
                  const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
                  v[c][0] = t.x; v[c][1] = t.y; v[c][2] = t.z; v[c][3] = t.w;
                } else {
                  const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
                  v[c][0] = t.x; v[c][1] = t.y;
                }
              }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              if (cb + c < x.nchunks) {
                const float w = mw[hh * 16 + cb + c];
#pragma unroll
                for (int e = 0; e < VW; ++e) o[e] = fmaf(v[c][e], w, o[e]);
              }
            }
          }
#pragma unroll
          for (int e = 0; e < VW; ++e) orow[hh * D + VW * lane + e] = MV<T>::from_f(o[e]);
        }
        __syncwarp();
      }
    }
  }
  cp_async_wait_group<0>();  // every copy this warp issued was consumed; drain regardless
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
  cfg.dynamicSmemBytes = S::smem_bytes(p.batch, p.ids_cap);
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

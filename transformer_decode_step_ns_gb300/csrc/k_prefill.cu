// Causal attention of a prefill chunk: the rows of one prompt chunk, at consecutive positions
// p0 .. p0 + C - 1 over one block table, each attending to every cached token up to its own
// position.  "NanoFlow ..." ("Four resource classes"): prefill attention is the compute-bound
// member of the attention class; the chunk rows of a dense batch (the pages' constant-size
// batches top up decode with chunked prefill) read the same K/V prefix, so this kernel reads
// each K/V block once per 16 queries and every q head of the group instead of once per row.
//
// CTA = (16-query tile, kv head g); warp w takes q head g * G + w for the 16 queries:
//   S[query][token]  = Q[query][:] . K[token][:]     (A = Q in registers, B = K tile, ldmatrix)
//   O[query][dim]   += P[query][token] . V[token][dim] (A = P from the S accumulator, B = V tile
//                                                       through ldmatrix.trans)
// with an online softmax per query row in the log2 domain.  K/V tiles stream through a
// cp.async ring shared by the CTA's warps.  Blocks are visited in order and every query row is
// reduced by one warp, so a row's result does not depend on how the chunk is tiled or split
// across nano-batches.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ns_internal.h"
#include "ns_ptx.cuh"

namespace ns {

namespace {

template <typename T>
struct PV;
template <>
struct PV<__half> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
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
struct PV<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace

template <int D>
struct PrefillShape {
  static constexpr int BS = 16;              // tokens per cache block
  static constexpr int TILE = BS * D * 2;    // bytes of one K or V tile
  static constexpr int STAGE = 2 * TILE;     // K then V
  static constexpr int NST = 3;              // ring depth
  static constexpr int KS = D / 16;          // QK k-steps
  static constexpr int NT = D / 8;           // PV n-tiles (8 dims each)
};

// Tile layout in shared memory: row t (token) of 128-byte halves h; 16-byte chunk cc of a half
// is stored at h * BS * 128 + t * 128 + ((cc ^ (t & 7)) << 4), which keeps ldmatrix conflict free.
template <typename T, int D, int G>
__global__ void __launch_bounds__(32 * G) prefill_attn_kernel(const PrefillParams p) {
  using S = PrefillShape<D>;
  __shared__ __align__(128) uint8_t ring[S::NST * S::STAGE];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Grid (kv heads, query tiles), launched in that order: every head's longest tile first (the
  // work of a tile grows with its position along the causal triangle), so the short ones fill
  // the tail.  q0 is the tile's first query (chunk-relative).
  const int q0 = (gridDim.y - 1 - blockIdx.y) * 16;
  const int g = blockIdx.x;
  const int h = g * G + warp;      // this warp's q head
  const int Hkv = p.n_kv_heads;
  griddep_wait();  // q and the chunk's K/V come from the QKV projection of this step
  if (tid == 0) griddep_launch_dependents();
  const int p0 = p.positions[p.row0];
  const int n_q = min(16, p.chunk - q0);
  const int last_pos = p0 + q0 + n_q - 1;  // the tile's last query position
  const int nblk = last_pos / S::BS + 1;
  const int* table = p.block_tables + static_cast<size_t>(p.row0) * p.mb;
  const T* kpool = reinterpret_cast<const T*>(p.k_pool);
  const T* vpool = reinterpret_cast<const T*>(p.v_pool);

  auto issue = [&](int blk) {
    if (blk < nblk) {
      int id = table[blk];
      if (id < 0 || id >= p.num_blocks) {
        if (tid == 0) atomicCAS(p.err, 0, NS_DEV_BAD_BLOCK);
        id = 0;
      }
      const size_t off = (static_cast<size_t>(id) * Hkv + g) * S::BS * D;
      const uint8_t* ks = reinterpret_cast<const uint8_t*>(kpool + off);
      const uint8_t* vs = reinterpret_cast<const uint8_t*>(vpool + off);
      const uint32_t dst = smem_u32(ring + (blk % S::NST) * S::STAGE);
      for (int c = tid; c < 2 * S::BS * D / 8; c += 32 * G) {
        const int kv = c / (S::BS * D / 8), ci = c - kv * (S::BS * D / 8);
        const int t = ci / (D / 8), c16 = ci % (D / 8);
        const int hh = c16 >> 3, cc = c16 & 7;
        const uint32_t d_off = kv * S::TILE + hh * (S::BS * 128) + t * 128 + ((cc ^ (t & 7)) << 4);
        cp16(dst + d_off, (kv ? vs : ks) + ci * 16);
      }
    }
    cp_commit();
  };

  // Q fragment of the 16 queries (A operand, row-major 16 x 16 per k-step); rows past the chunk
  // read as zeros
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t qa[S::KS][4];
  {
    const T* qb = reinterpret_cast<const T*>(p.q);
    const bool v0 = gq < n_q, v1 = gq + 8 < n_q;
    const T* r0 = qb + (static_cast<size_t>(p.row0 + q0 + gq) * p.q_row_stride) + static_cast<size_t>(h) * D;
    const T* r1 = r0 + 8 * p.q_row_stride;
#pragma unroll
    for (int ks = 0; ks < S::KS; ++ks) {
      const int c = ks * 16 + 2 * tq;
      qa[ks][0] = v0 ? *reinterpret_cast<const uint32_t*>(r0 + c) : 0u;
      qa[ks][1] = v1 ? *reinterpret_cast<const uint32_t*>(r1 + c) : 0u;
      qa[ks][2] = v0 ? *reinterpret_cast<const uint32_t*>(r0 + c + 8) : 0u;
      qa[ks][3] = v1 ? *reinterpret_cast<const uint32_t*>(r1 + c + 8) : 0u;
    }
  }

  float acc[S::NT][4];
#pragma unroll
  for (int n = 0; n < S::NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gq and gq + 8
  const int qp0 = p0 + q0 + gq, qp1 = qp0 + 8;                // their positions
  // ldmatrix lanes: K (B operand of QK): matrices (tokens 0-7 | 8-15) x (chunk c | c + 1)
  const int k_tok = (lane & 7) + ((lane >> 4) << 3), k_chk = (lane >> 3) & 1;
  // V (B operand of PV, transposed): matrices (tokens 0-7, 8-15) x (chunk c, c + 1)
  const int v_tok = (lane & 7) + (((lane >> 3) & 1) << 3), v_chk = lane >> 4;

  for (int s = 0; s < S::NST - 1; ++s) issue(s);
  for (int blk = 0; blk < nblk; ++blk) {
    issue(blk + S::NST - 1);
    cp_wait<S::NST - 1>();
    __syncthreads();
    const uint32_t kbase = smem_u32(ring + (blk % S::NST) * S::STAGE);
    const uint32_t vbase = kbase + S::TILE;
    // ---- S = Q K^T for tokens blk * 16 .. + 15 (two n-tiles of 8)
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < S::KS; ++ks) {
      const int c16 = 2 * ks + k_chk;
      const int hh = c16 >> 3, cc = c16 & 7;
      uint32_t kb[4];
      ldsm4(kbase + hh * (S::BS * 128) + k_tok * 128 + ((cc ^ (k_tok & 7)) << 4), kb);
      PV<T>::mma(sacc[0], qa[ks], kb[0], kb[1]);
      PV<T>::mma(sacc[1], qa[ks], kb[2], kb[3]);
    }
    // ---- causal mask and online softmax per query row
    float x[2][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const int kp = blk * S::BS + n * 8 + 2 * tq;
      x[n][0] = kp <= qp0 ? sacc[n][0] * p.scale_log2 : -INFINITY;
      x[n][1] = kp + 1 <= qp0 ? sacc[n][1] * p.scale_log2 : -INFINITY;
      x[n][2] = kp <= qp1 ? sacc[n][2] * p.scale_log2 : -INFINITY;
      x[n][3] = kp + 1 <= qp1 ? sacc[n][3] * p.scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(x[n][0], x[n][1]));
      mx1 = fmaxf(mx1, fmaxf(x[n][2], x[n][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // a row with every token masked so far keeps m = -inf; use 0 as its exponent base
    const float b0 = n0 == -INFINITY ? 0.f : n0, b1 = n1 == -INFINITY ? 0.f : n1;
    const float a0 = exp2f(m0 - b0), a1 = exp2f(m1 - b1);
    float pr[2][4], s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      pr[n][0] = exp2f(x[n][0] - b0);
      pr[n][1] = exp2f(x[n][1] - b0);
      pr[n][2] = exp2f(x[n][2] - b1);
      pr[n][3] = exp2f(x[n][3] - b1);
      s0 += pr[n][0] + pr[n][1];
      s1 += pr[n][2] + pr[n][3];
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    l0 = l0 * a0 + s0;
    l1 = l1 * a1 + s1;
    m0 = n0;
    m1 = n1;
    // ---- O = O * alpha + P V  (P as the A operand straight from the S accumulator layout)
    const uint32_t pa[4] = {PV<T>::pack(pr[0][0], pr[0][1]), PV<T>::pack(pr[0][2], pr[0][3]),
                            PV<T>::pack(pr[1][0], pr[1][1]), PV<T>::pack(pr[1][2], pr[1][3])};
#pragma unroll
    for (int n = 0; n < S::NT; ++n) {
      acc[n][0] *= a0;
      acc[n][1] *= a0;
      acc[n][2] *= a1;
      acc[n][3] *= a1;
    }
#pragma unroll
    for (int n2 = 0; n2 < S::NT / 2; ++n2) {
      const int c16 = 2 * n2 + v_chk;
      const int hh = c16 >> 3, cc = c16 & 7;
      uint32_t vb[4];
      ldsm4_t(vbase + hh * (S::BS * 128) + v_tok * 128 + ((cc ^ (v_tok & 7)) << 4), vb);
      PV<T>::mma(acc[2 * n2], pa, vb[0], vb[1]);
      PV<T>::mma(acc[2 * n2 + 1], pa, vb[2], vb[3]);
    }
    __syncthreads();  // the stage is refilled by the next iteration's issue
  }
  cp_wait<0>();

  // ---- O / l, stored for the tile's valid rows
  T* out = reinterpret_cast<T*>(p.out);
  const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
  for (int n = 0; n < S::NT; ++n) {
    const int d = n * 8 + 2 * tq;
    if (gq < n_q) {
      T* o = out + static_cast<size_t>(p.row0 + q0 + gq) * p.out_row_stride + static_cast<size_t>(h) * D + d;
      *reinterpret_cast<uint32_t*>(o) = PV<T>::pack(acc[n][0] * i0, acc[n][1] * i0);
    }
    if (gq + 8 < n_q) {
      T* o = out + static_cast<size_t>(p.row0 + q0 + gq + 8) * p.out_row_stride + static_cast<size_t>(h) * D + d;
      *reinterpret_cast<uint32_t*>(o) = PV<T>::pack(acc[n][2] * i1, acc[n][3] * i1);
    }
  }
}

// ------------------------------------------------------------------------------ host side

namespace {

template <typename T, int D, int G>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_kv_heads, (p.chunk + 15) / 16, 1);
  cfg.blockDim = dim3(32 * G, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prefill_attn_kernel<T, D, G>, p);
}

template <typename T, int D>
cudaError_t prefill_g(const PrefillParams& p, int group, cudaStream_t s, bool pdl) {
  switch (group) {
    case 1: return launch_prefill_t<T, D, 1>(p, s, pdl);
    case 2: return launch_prefill_t<T, D, 2>(p, s, pdl);
    case 4: return launch_prefill_t<T, D, 4>(p, s, pdl);
    case 7: return launch_prefill_t<T, D, 7>(p, s, pdl);
    case 8: return launch_prefill_t<T, D, 8>(p, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, int dtype, int head_dim, int group,
                           cudaStream_t s, bool pdl) {
  if (p.chunk < 1) return cudaSuccess;
  if (dtype == NS_BF16)
    return head_dim == 64 ? prefill_g<__nv_bfloat16, 64>(p, group, s, pdl)
                          : prefill_g<__nv_bfloat16, 128>(p, group, s, pdl);
  return head_dim == 64 ? prefill_g<__half, 64>(p, group, s, pdl)
                        : prefill_g<__half, 128>(p, group, s, pdl);
}

}  // namespace ns

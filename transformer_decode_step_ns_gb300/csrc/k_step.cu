// Persistent decode step for small batches: one cooperative launch runs the whole step.
//
// "The chef who calls out every order" / "The maths that matters: when the GPU is left waiting"
// (nanoserve notes): at small batch a decode step is a long chain of short dependent kernels,
// each paying a launch and a dependency wait that are larger than its own weight read.  Here
// the chain runs inside one kernel with one CTA per SM:
//
// * One warp per CTA streams that CTA's share of every layer's weights (and then the LM head's)
//   through a ring of 16 KiB shared-memory slots (four 4 KiB chunks) with 1-D TMA bulk copies.  The weights do not
//   depend on the activations, so the stream never waits on the stage chain: the next stages'
//   weights are in shared memory when their inputs become ready.  The shares are packed once
//   (ns_set_step_kernel) into one contiguous stream per CTA, in the order they are consumed,
//   already in the register layout of the tensor-core operands.
// * Seven compute warps run the stages: embedding + RoPE table, then per layer QKV (RMSNorm
//   scale, RoPE, q store, paged K/V write), attention, O (+ residual, next norm's inputs),
//   gate/up (+ SwiGLU), down (+ residual, next norm's inputs), and finally the LM head.  Stages
//   are separated by a grid-wide barrier (an arrival counter, release/acquire at GPU scope, the
//   one-second %globaltimer limit of every wait in this library).
// * Projection stages: a 16-feature output tile times the batch (padded to 8-row n-tiles) is a
//   chain of mma.sync m16n8k16 products with the weight tile as A.  At these batch sizes the
//   projections read their weights once at 2B flop per weight ("The roofline flips": AI ~ 2B),
//   far below any tensor pipe's ridge, so what counts is streaming the weights and the latency
//   of each stage, not tcgen05 throughput.  A stage first copies the activation columns it
//   reduces over, for every row, into shared memory with one bulk copy (activations are stored
//   in 128-column chunks [chunk][row][128], so any column range of all rows is contiguous; all
//   CTAs read the same activation at once, which one TMA request per CTA serves several times
//   faster than per-lane loads).  Warp w takes the 128-column chunks w, w + 7, ... of every tile
//   of the CTA, and the warps' partial tiles are summed in warp order.  Reductions longer than
//   kStepSliceChunks chunks are split over teams of CTAs; each split's partial tile goes to
//   global memory and the member that finishes a tile last sums the splits in split order and
//   runs the epilogue.  Within a 32-column block the reduction index is permuted so that each
//   lane's operand is 8 consecutive columns of a row (one 16-byte load); the weights are packed
//   with the same permutation, so the dot products are unchanged.
// * Attention unit = (row, kv head, 14 cache blocks): each warp takes one or two blocks, the
//   G query heads of the group are the rows of one m16 tile (S = q K^T with K straight from
//   global memory, O^T += V^T P^T with V staged through shared memory), online softmax in the
//   log2 domain; the warps' results are merged in warp order, and the units of a row by the CTA
//   that finishes last (atomic counter) in unit order.
// * Every reduction order depends on the weight shapes and the row's own length only, so a
//   row's result does not depend on the rest of the batch or on which CTA computes it.
//
// Data written inside the kernel and read by another CTA is read with ld.global.cg (L2), never
// through L1, which is not coherent across SMs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "ns_epi.cuh"
#include "ns_host.h"
#include "ns_internal.h"
#include "ns_ptx.cuh"

namespace ns {

namespace {

template <typename T>
struct SV;
template <>
struct SV<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
};
template <>
struct SV<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
};

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The streaming warp publishes how many chunks it has issued with a CTA-scope release; a
// consumer that reads the count with an acquire also sees the slot barrier's earlier phases.
__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void cp_async_16_cg(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_commit_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Shared-memory control block of a CTA.
struct StepCtl {
  int issued;  // chunks the streaming warp has issued
  int abort;   // this CTA stops (a wait ran out, or another CTA stopped)
  int flag;    // CTA-uniform decisions
  int pad;
};

// Everything a compute warp needs about its CTA.
struct Ctx {
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* actbar;   // completion of the stage's activation copy
  StepCtl* ctl;
  float* rs;          // [kStepMaxRows] RMSNorm scales of the current stage
  int* prefix;        // [kStepMaxRows + 1] attention unit offsets per row
  int* s_seq;         // [kStepMaxRows] step metadata copied once
  long long* s_slot;  // [kStepMaxRows]
  int* last;          // [kStepMaxTilesPerCta] split-K tiles this CTA finishes
  float* s_cos;       // [kStepMaxRows][D / 2] RoPE table of the step's rows
  float* s_sin;
  uint8_t* act;       // kStepActBytes: the stage's activation columns
  float* red;         // warps' partial tiles
  uint8_t* stage;     // attention staging (over act and red)
  int warp, lane, tid;
  unsigned gen;       // grid barriers passed
  int seq;            // next chunk of this CTA's stream
  int actn;           // activation copies so far (the phase of actbar)
  int early_ok;       // the step writes no block that a row reads before its last
  int rows_valid;
  float* logits;
};

__device__ __forceinline__ bool cta_aborted(const Ctx& cx) {
  return *reinterpret_cast<volatile int*>(&cx.ctl->abort) != 0;
}

__device__ __forceinline__ void cta_abort(const Ctx& cx, const StepParams& p) {
  if (!cta_aborted(cx)) {
    *reinterpret_cast<volatile int*>(&cx.ctl->abort) = 1;
    set_err(p.err, NS_DEV_WAIT_TIMEOUT);
  }
}

// Wait until chunk `idx` of the stream is in shared memory.  The streaming warp issues chunks
// in order and reuses a slot only after its previous chunks were released, so once `issued`
// passes idx the slot's barrier is at most one phase behind and its parity names the right
// phase.
__device__ __forceinline__ bool wait_chunk(const Ctx& cx, const StepParams& p, int idx) {
  if (ld_acquire_cta(&cx.ctl->issued) <= idx) {
    const unsigned long long t0 = global_timer_ns();
    while (ld_acquire_cta(&cx.ctl->issued) <= idx) {
      if (cta_aborted(cx)) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        cta_abort(cx, p);
        return false;
      }
    }
  }
  const int blk = idx / kStepSlotChunks, s = blk % p.nslot;
  if (!mbar_wait(&cx.full[s], static_cast<uint32_t>(blk / p.nslot) & 1u, &cx.ctl->abort)) {
    cta_abort(cx, p);
    return false;
  }
  return true;
}

// Grid-wide barrier of the compute warps of every CTA: after a CTA barrier, thread 0 adds one
// arrival with a GPU-scope release and polls the count with GPU-scope acquires; the CTA barrier
// that follows passes what it acquired on to the CTA.  Activations written before the barrier
// are read afterwards by TMA (the async proxy), so every thread first orders its global and
// shared-memory accesses for the async proxy.  Returns false (uniformly within the CTA) when the step is abandoned.
__device__ bool grid_sync(Ctx& cx, const StepParams& p) {
  fence_proxy_async_global();
  fence_proxy_async_shared();  // the next stage's copy overwrites shared memory this one used
  named_barrier_sync(1, kStepWarps * 32);
  if (cx.tid == 0) {
    cx.gen += 1;
    const unsigned target = cx.gen * gridDim.x;
    int stop = cta_aborted(cx);
    red_release_gpu_add(&p.sync[0], 1u);
    if (!stop) {
      const unsigned long long t0 = global_timer_ns();
      for (uint32_t i = 0;; ++i) {
        if (ld_acquire_gpu(&p.sync[0]) >= target) break;
        if ((i & 15u) == 15u) {
          if (*reinterpret_cast<volatile unsigned*>(&p.sync[1]) != 0u) {
            stop = 1;
            break;
          }
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            set_err(p.err, NS_DEV_WAIT_TIMEOUT);
            stop = 1;
            break;
          }
        }
      }
    }
    if (stop) {
      atomicExch(&p.sync[1], 1u);
      *reinterpret_cast<volatile int*>(&cx.ctl->abort) = 1;
    }
    cx.ctl->flag = stop;
  }
  named_barrier_sync(1, kStepWarps * 32);
  // ctl->flag is written again only after the next CTA barrier, which every thread reaches
  // after this read
  return cx.ctl->flag == 0;
}

// Element (row, col) of a chunk-major activation [width / 128][B][128].
__device__ __forceinline__ size_t cm_index(int row, int col, int B) {
  return (static_cast<size_t>(col >> 7) * B + row) * 128 + (col & 127);
}

// ------------------------------------------------------------------ step set-up, embedding
// Copy the rows' lengths and slots into shared memory and build the RoPE table of the step's
// rows (every CTA builds its own; the positions are shared by all layers).
template <int D>
__device__ void step_setup(Ctx& cx, const StepParams& p) {
  constexpr int half = D / 2;
  if (cx.tid < p.B) {
    cx.s_seq[cx.tid] = p.seq[cx.tid];
    cx.s_slot[cx.tid] = p.slot[cx.tid];
  }
  for (int e = cx.tid; e < p.B * half; e += kStepWarps * 32) {
    const int tok = e / half, i = e - tok * half;
    rope_cos_sin(p.pos[tok], p.inv_freq[i], &cx.s_cos[e], &cx.s_sin[e]);
  }
  cx.early_ok = p.early_ok != nullptr ? *p.early_ok : 0;
  cx.rows_valid = *p.rows_valid;
  cx.logits = p.with_lm ? reinterpret_cast<float*>(*p.logits_slot) : nullptr;
}

template <typename T>
__device__ void embed_stage(const Ctx& cx, const StepParams& p) {
  const int H16 = p.H / 16;
  const int hw = cx.tid >> 4, hl = cx.tid & 15;
  const unsigned hmask = 0xffffu << (cx.lane & 16);
  const T* emb = reinterpret_cast<const T*>(p.embed);
  T* xn = reinterpret_cast<T*>(p.xn);
  for (int it = blockIdx.x * (kStepWarps * 2) + hw; it < p.B * H16; it += gridDim.x * (kStepWarps * 2)) {
    const int tok = it / H16, tt = it - tok * H16;
    const int f = tt * 16 + hl;
    int id = tok >= cx.rows_valid ? 0 : p.tok[tok];
    // -(r + 1): the token sampled at row r of the previous step, in the device token source
    if (id < 0 && p.tok_src != nullptr) id = p.tok_src[-id - 1];
    if (id < 0 || id >= p.vocab) {
      if (hl == 0 && tt == 0) set_err(p.err, NS_DEV_BAD_TOKEN);
      id = 0;
    }
    const float x = SV<T>::to_f(emb[static_cast<size_t>(id) * p.H + f]);
    p.resid[static_cast<size_t>(tok) * p.H + f] = x;
    xn[cm_index(tok, f, p.B)] = SV<T>::from_f(x * p.attn_norm[f]);
    float s = x * x;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(hmask, s, o);
    if (hl == 0) p.sumsq16[tok * H16 + tt] = s;
  }
}

// rs[tok] = 1 / sqrt(mean of squares + eps) of every row, from the per-16-column partial sums
// the stage copied into shared memory ([row][H / 16]): lanes over the partials, a fixed shuffle
// tree (the order depends on H only).
__device__ void row_scales(const Ctx& cx, const StepParams& p, const float* sums) {
  const int n16 = p.H / 16;
  for (int tok = cx.warp; tok < p.B; tok += kStepWarps) {
    float x = 0.f;
    for (int t = cx.lane; t < n16; t += 32) x += sums[tok * n16 + t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (cx.lane == 0) cx.rs[tok] = rms_scale(x, p.H, p.eps);
  }
}

// ------------------------------------------------------------------ projection stages
// acc[ti] += chunk(idx0 + ti) x bx for the tiles of one group
template <typename T>
__device__ __forceinline__ void chunk_products(const Ctx& cx, const StepParams& p, int idx0, int tg, int NT,
                                               const uint4 (&bx)[4][4], float (&acc)[kStepGroup][4][4]) {
#pragma unroll
  for (int ti = 0; ti < kStepGroup; ++ti) {
    if (ti >= tg) break;
    const int idx = idx0 + ti;
    if (!wait_chunk(cx, p, idx)) continue;
    const int slot = (idx / kStepSlotChunks) % p.nslot;
    const uint8_t* ch = cx.ring + static_cast<size_t>(slot) * kStepSlot + (idx % kStepSlotChunks) * kStepChunk;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint4 a = *reinterpret_cast<const uint4*>(ch + ((kp * 2 + h2) * 32 + cx.lane) * 16);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          if (nt < NT) {
            const uint32_t b0 = h2 ? bx[kp][nt].z : bx[kp][nt].x;
            const uint32_t b1 = h2 ? bx[kp][nt].w : bx[kp][nt].y;
            SV<T>::mma(acc[ti][nt], a.x, a.y, a.z, a.w, b0, b1);
          }
        }
      }
    __syncwarp();
    if (cx.lane == 0) mbar_arrive(&cx.empty[slot]);
  }
}

// The epilogue of one (tile, row, feature pair fp / fp + 8) of a projection with the summed
// products lo, hi.  pre, when given, holds the residual and gain of a residual stage (loaded
// ahead).  Residual stages shuffle across the 8 lanes of a row: call them warp-uniformly.
template <typename T, int D>
__device__ __forceinline__ void epilogue(const Ctx& cx, const StepParams& p, int kind, int layer, int tt,
                                         int tok, int fp, float lo, float hi, const float* pre) {
  const bool live = tok < p.B;
  if (kind == SS_O || kind == SS_DOWN) {
    // resid += y; next norm's input x * gamma; this tile's sum of squares per row
    const float* gam = kind == SS_O ? p.ffn_norm + static_cast<size_t>(layer) * p.H
                       : layer + 1 < p.n_layers ? p.attn_norm + static_cast<size_t>(layer + 1) * p.H
                                                : p.final_norm;
    const int n_lo = tt * 16 + fp, n_hi = n_lo + 8;
    float r_lo = 0.f, r_hi = 0.f;
    if (live) {
      float* rrow = p.resid + static_cast<size_t>(tok) * p.H;
      const float o_lo = pre ? pre[0] : __ldcg(&rrow[n_lo]);
      const float o_hi = pre ? pre[1] : __ldcg(&rrow[n_hi]);
      const float g_lo = pre ? pre[2] : gam[n_lo];
      const float g_hi = pre ? pre[3] : gam[n_hi];
      r_lo = o_lo + lo;
      r_hi = o_hi + hi;
      rrow[n_lo] = r_lo;
      rrow[n_hi] = r_hi;
      T* xn = reinterpret_cast<T*>(p.xn);
      xn[cm_index(tok, n_lo, p.B)] = SV<T>::from_f(r_lo * g_lo);
      xn[cm_index(tok, n_hi, p.B)] = SV<T>::from_f(r_hi * g_hi);
    }
    float sq = r_lo * r_lo + r_hi * r_hi;
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    sq += __shfl_xor_sync(0xffffffffu, sq, 4);
    if (live && fp == 0) p.sumsq16[tok * (p.H / 16) + tt] = sq;
    return;
  }
  if (!live) return;
  const float sc = cx.rs[tok];
  if (kind == SS_GU) {
    reinterpret_cast<T*>(p.act)[cm_index(tok, tt * 8 + fp, p.B)] = SV<T>::from_f(silu_mul(lo * sc, hi * sc));
  } else if (kind == SS_LM) {
    if (tok >= cx.rows_valid) return;  // padding rows of a bucketed graph have no output row
    float* out = cx.logits + static_cast<size_t>(tok) * p.vocab;
    out[tt * 16 + fp] = lo * sc;
    out[tt * 16 + fp + 8] = hi * sc;
  } else {  // SS_QKV: RoPE pairs (i, i + d/2) of q/k heads, plain v columns
    constexpr int dh = D / 16, half = D / 2;
    const int nrope = (p.Hq + p.Hkv) * dh;
    const long long slot = cx.s_slot[tok];
    auto kv_off = [&](int kvh) {
      return ((static_cast<size_t>(slot / p.block_size) * p.Hkv + kvh) * p.block_size +
              static_cast<size_t>(slot % p.block_size)) * D;
    };
    if (tt >= p.Hq * dh && (slot < 0 || slot >= p.pool_slots)) {
      set_err(p.err, NS_DEV_BAD_SLOT);
      return;
    }
    if (tt < nrope) {
      const int hh = tt / dh, i = (tt - hh * dh) * 8 + fp;
      const float c = cx.s_cos[tok * half + i], sn = cx.s_sin[tok * half + i];
      const float x_lo = lo * sc, x_hi = hi * sc;
      const float y_lo = rope_lo(x_lo, x_hi, c, sn), y_hi = rope_hi(x_lo, x_hi, c, sn);
      if (hh < p.Hq) {
        T* qo = reinterpret_cast<T*>(p.q) + static_cast<size_t>(tok) * p.qd + hh * D;
        qo[i] = SV<T>::from_f(y_lo);
        qo[i + half] = SV<T>::from_f(y_hi);
      } else {
        T* kp = reinterpret_cast<T*>(p.pools + static_cast<size_t>(2 * layer) * p.pool_bytes) + kv_off(hh - p.Hq);
        kp[i] = SV<T>::from_f(y_lo);
        kp[i + half] = SV<T>::from_f(y_hi);
      }
    } else {
      T* vp = reinterpret_cast<T*>(p.pools + static_cast<size_t>(2 * layer + 1) * p.pool_bytes);
      const int f_lo = (tt - nrope) * 16 + fp, f_hi = f_lo + 8;
      vp[kv_off(f_lo / D) + f_lo % D] = SV<T>::from_f(lo * sc);
      vp[kv_off(f_hi / D) + f_hi % D] = SV<T>::from_f(hi * sc);
    }
  }
}

template <typename T, int D>
__device__ void gemm_stage(Ctx& cx, const StepParams& p, int kind, int layer) {
  constexpr int kItems = (kStepGroup * kStepMaxRows * 8 + kStepWarps * 32 - 1) / (kStepWarps * 32);
  const StepTiles st = step_tiles(gridDim.x, blockIdx.x, p.n_tiles[kind], p.kc[kind], p.split[kind], p.rot[kind]);
  const int S = p.split[kind];
  const int nkc = st.kc1 - st.kc0;
  const int NT = (p.B + 7) >> 3, Bp = NT * 8;
  const int g = cx.lane >> 2, t = cx.lane & 3;
  const bool resid_kind = kind == SS_O || kind == SS_DOWN;
  if (st.count == 0) return;  // uniform: no chunks, no copy, no barrier
  // the activation columns [kc0, kc1) of every row: one bulk copy
  // (stages that apply the RMSNorm scale also copy the rows' sums of squares, into the space of
  // the partial tiles, which they use only after the scales are computed)
  const bool scaled = kind == SS_QKV || kind == SS_GU || kind == SS_LM;
  if (cx.tid == 0) {
    const T* src = reinterpret_cast<const T*>(kind == SS_O ? p.o : kind == SS_DOWN ? p.act : p.xn) +
                   static_cast<size_t>(st.kc0) * p.B * 128;
    const uint32_t bytes = static_cast<uint32_t>(nkc) * p.B * 256;
    const uint32_t sbytes = scaled ? static_cast<uint32_t>(p.B) * (p.H / 16) * 4 : 0u;
    fence_proxy_async_shared();  // the region's earlier generic accesses precede the copy
    mbar_arrive_expect_tx(cx.actbar, bytes + sbytes);
    bulk_g2s(cx.act, src, bytes, cx.actbar);
    if (scaled) bulk_g2s(cx.red, p.sumsq16, sbytes, cx.actbar);
  }
  // residual-stage epilogue inputs of the first group, loaded while the copy and products run
  float pre[kItems][4];
  if (resid_kind && S == 1) {
    const int tg = min(kStepGroup, st.count);
    const float* gam = kind == SS_O ? p.ffn_norm + static_cast<size_t>(layer) * p.H
                       : layer + 1 < p.n_layers ? p.attn_norm + static_cast<size_t>(layer + 1) * p.H
                                                : p.final_norm;
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int it = cx.tid + k * kStepWarps * 32;
      const int ti = it / (Bp * 8), tok = (it >> 3) % Bp, fp = it & 7;
      pre[k][0] = pre[k][1] = pre[k][2] = pre[k][3] = 0.f;
      if (it < tg * Bp * 8 && tok < p.B) {
        const int n_lo = (st.first + ti * st.stride) * 16 + fp;
        const float* rrow = p.resid + static_cast<size_t>(tok) * p.H;
        pre[k][0] = __ldcg(&rrow[n_lo]);
        pre[k][1] = __ldcg(&rrow[n_lo + 8]);
        pre[k][2] = gam[n_lo];
        pre[k][3] = gam[n_lo + 8];
      }
    }
  }
  const bool act_ok = mbar_wait(cx.actbar, static_cast<uint32_t>(cx.actn) & 1u, &cx.ctl->abort);
  cx.actn += 1;
  if (!act_ok) cta_abort(cx, p);
  if (scaled) {
    if (act_ok) row_scales(cx, p, cx.red);
    named_barrier_sync(1, kStepWarps * 32);  // the sums are read before partial tiles overwrite them
  }
  for (int g0 = 0; g0 < st.count; g0 += kStepGroup) {
    const int tg = min(kStepGroup, st.count - g0);
    float acc[kStepGroup][4][4];
#pragma unroll
    for (int a = 0; a < kStepGroup; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;
    if (act_ok) {
      for (int kcl = cx.warp; kcl < nkc; kcl += kStepWarps) {
        // lane (g, t): columns 32 kp + 8 t .. + 7 of row nt * 8 + g of local chunk kcl
        uint4 bx[4][4];
#pragma unroll
        for (int kp = 0; kp < 4; ++kp)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const int row = nt * 8 + g;
            bx[kp][nt] = make_uint4(0u, 0u, 0u, 0u);
            if (nt < NT && row < p.B)
              bx[kp][nt] = *reinterpret_cast<const uint4*>(cx.act + ((kcl * p.B + row) * 128 + kp * 32 + 8 * t) * 2);
          }
        chunk_products<T>(cx, p, cx.seq + kcl * tg, tg, NT, bx, acc);
      }
    }
    cx.seq += nkc * tg;
    // partial tiles -> shared memory [warp][tile][token][feature]
#pragma unroll
    for (int ti = 0; ti < kStepGroup; ++ti) {
      if (ti >= tg) break;
      float* rw = cx.red + (cx.warp * kStepGroup + ti) * kStepMaxRows * kStepRedStride;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        if (nt < NT) {
          const int tk = nt * 8 + 2 * t;
          rw[tk * kStepRedStride + g] = acc[ti][nt][0];
          rw[(tk + 1) * kStepRedStride + g] = acc[ti][nt][1];
          rw[tk * kStepRedStride + g + 8] = acc[ti][nt][2];
          rw[(tk + 1) * kStepRedStride + g + 8] = acc[ti][nt][3];
        }
      }
    }
    named_barrier_sync(1, kStepWarps * 32);
    // sum the warps' partials in warp order; thread -> (tile, token, feature pair f, f + 8)
    const int nw = min(kStepWarps, nkc);
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int it = cx.tid + k * kStepWarps * 32;
      if (it >= tg * Bp * 8) break;  // uniform per warp (the count and the stride are multiples of 32)
      const int ti = it / (Bp * 8), tok = (it >> 3) % Bp, fp = it & 7;
      float lo = 0.f, hi = 0.f;
      for (int w = 0; w < nw; ++w) {
        const float* rw = cx.red + ((w * kStepGroup + ti) * kStepMaxRows + tok) * kStepRedStride;
        lo += rw[fp];
        hi += rw[fp + 8];
      }
      const int tt = st.first + (g0 + ti) * st.stride;
      if (S == 1) {
        epilogue<T, D>(cx, p, kind, layer, tt, tok, fp, lo, hi, resid_kind && g0 == 0 ? pre[k] : nullptr);
      } else if (tok < p.B) {
        float* pt = p.split_part + ((static_cast<size_t>(tt) * S + st.split) * kStepMaxRows + tok) * 16;
        pt[fp] = lo;
        pt[fp + 8] = hi;
      }
    }
    named_barrier_sync(1, kStepWarps * 32);
  }
  if (S == 1) return;
  // split-K: the team member that completes a tile last sums its splits in split order and
  // runs the epilogue
  __threadfence();
  named_barrier_sync(1, kStepWarps * 32);
  if (cx.tid < st.count) {
    const int tt = st.first + cx.tid * st.stride;
    unsigned* cnt = p.sync + 2 + static_cast<size_t>(p.n_layers) * kStepMaxRows * p.Hkv +
                    (static_cast<size_t>(layer) * 4 + (kind == SS_LM ? 0 : kind)) * p.max_split_tiles + tt;
    cx.last[cx.tid] = atomicAdd(cnt, 1u) + 1 == static_cast<unsigned>(S);
  }
  named_barrier_sync(1, kStepWarps * 32);
  __threadfence();
  const float* gam = kind == SS_O ? p.ffn_norm + static_cast<size_t>(layer) * p.H
                     : layer + 1 < p.n_layers ? p.attn_norm + static_cast<size_t>(layer + 1) * p.H
                                              : p.final_norm;
  for (int ti = 0; ti < st.count; ++ti) {
    if (!cx.last[ti]) continue;  // uniform
    const int tt = st.first + ti * st.stride;
    for (int it = cx.tid; it < Bp * 8; it += kStepWarps * 32) {  // warp-uniform trip count
      const int tok = it >> 3, fp = it & 7;
      float v[8][2], in[4] = {0.f, 0.f, 0.f, 0.f};
      // the splits' partials and the residual inputs: every load issued before any is used
#pragma unroll
      for (int sp = 0; sp < 8; ++sp) {
        v[sp][0] = v[sp][1] = 0.f;
        if (sp < S && tok < p.B) {
          const float* pt = p.split_part + ((static_cast<size_t>(tt) * S + sp) * kStepMaxRows + tok) * 16;
          v[sp][0] = __ldcg(&pt[fp]);
          v[sp][1] = __ldcg(&pt[fp + 8]);
        }
      }
      if (resid_kind && tok < p.B) {
        const int n_lo = tt * 16 + fp;
        const float* rrow = p.resid + static_cast<size_t>(tok) * p.H;
        in[0] = __ldcg(&rrow[n_lo]);
        in[1] = __ldcg(&rrow[n_lo + 8]);
        in[2] = gam[n_lo];
        in[3] = gam[n_lo + 8];
      }
      float lo = 0.f, hi = 0.f;
#pragma unroll
      for (int sp = 0; sp < 8; ++sp) {
        lo += v[sp][0];
        hi += v[sp][1];
      }
      epilogue<T, D>(cx, p, kind, layer, tt, tok, fp, lo, hi, resid_kind ? in : nullptr);
    }
  }
  named_barrier_sync(1, kStepWarps * 32);
}

// ------------------------------------------------------------------ attention stage
// Unit u of the step: row b, kv head h, the 16-block range c of the row.
struct AttnUnit {
  int b, h, c, L, nbk, nch, jb, nblk;
};

__device__ __forceinline__ AttnUnit attn_unit(const Ctx& cx, const StepParams& p, int u) {
  AttnUnit a;
  a.b = 0;
  while (a.b + 1 < p.B && cx.prefix[a.b + 1] <= u) ++a.b;
  a.L = cx.s_seq[a.b];
  a.nbk = (a.L + 15) >> 4;
  a.nch = (a.nbk + kStepAttnBlocks - 1) / kStepAttnBlocks;
  const int r = u - cx.prefix[a.b];
  a.h = r / a.nch;
  a.c = r - a.h * a.nch;
  a.jb = a.c * kStepAttnBlocks + cx.warp;  // this warp's first block; its second is jb + kStepWarps
  a.nblk = a.jb < a.nbk ? (a.jb + kStepWarps < a.nbk ? 2 : 1) : 0;
  return a;
}

template <typename T, int D>
struct AttnFetch {
  uint2 kr[2][D / 16][2];  // K operands of the warp's two blocks
  int u;                   // the unit whose blocks were fetched before the barrier (-1: none)
  bool done[2];            // block bi of unit u is already fetched
};

// Fetch K (registers) and V (staged in shared memory) of block bi of unit a.
template <typename T, int D>
__device__ __forceinline__ void attn_fetch_block(const Ctx& cx, const StepParams& p, int layer,
                                                 const AttnUnit& a, int bi, AttnFetch<T, D>& f) {
  constexpr int KS = D / 16, VROW = (D + 8) * 2, VBLK = 16 * VROW;
  const int g = cx.lane >> 2, t = cx.lane & 3;
  const T* kpool = reinterpret_cast<const T*>(p.pools + static_cast<size_t>(2 * layer) * p.pool_bytes);
  const T* vpool = reinterpret_cast<const T*>(p.pools + static_cast<size_t>(2 * layer + 1) * p.pool_bytes);
  int phys = p.tab[static_cast<size_t>(a.b) * p.mb + a.jb + kStepWarps * bi];
  if (phys < 0 || phys >= p.num_blocks) {
    set_err(p.err, NS_DEV_BAD_BLOCK);
    phys = 0;
  }
  const size_t base = (static_cast<size_t>(phys) * p.Hkv + a.h) * 16 * D;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
      f.kr[bi][ks][nt] = __ldcg(reinterpret_cast<const uint2*>(kpool + base + (nt * 8 + g) * D + 16 * ks + 4 * t));
  uint8_t* vst = cx.stage + cx.warp * 2 * VBLK + bi * VBLK;
  const T* vb = vpool + base;
#pragma unroll
  for (int i = cx.lane; i < 16 * D / 8; i += 32) {
    const int row = i / (D / 8), c8 = i - row * (D / 8);
    cp_async_16_cg(smem_u32(vst + row * VROW + c8 * 16), vb + row * D + c8 * 8);
  }
}

// Before the barrier that ends the QKV stage: the unit offsets, and the first unit's blocks
// other than its row's last (the only block this step writes, when early_ok) are fetched, so
// their latency overlaps the barrier.
template <typename T, int D>
__device__ void attn_prepare(Ctx& cx, const StepParams& p, int layer, AttnFetch<T, D>& f) {
  if (cx.warp == 0) {
    int u = 0;
    if (cx.lane < p.B) {
      const int nbk = (cx.s_seq[cx.lane] + 15) >> 4;
      u = p.Hkv * ((nbk + kStepAttnBlocks - 1) / kStepAttnBlocks);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, u, o);
      if (cx.lane >= o) u += v;
    }
    if (cx.lane < p.B) cx.prefix[cx.lane + 1] = u;
    if (cx.lane == 0) cx.prefix[0] = 0;
  }
  named_barrier_sync(1, kStepWarps * 32);
  f.u = -1;
  f.done[0] = f.done[1] = false;
  if (!cx.early_ok || static_cast<int>(blockIdx.x) >= cx.prefix[p.B]) return;
  f.u = blockIdx.x;
  const AttnUnit a = attn_unit(cx, p, f.u);
#pragma unroll
  for (int bi = 0; bi < 2; ++bi) {
    if (bi < a.nblk && a.jb + kStepWarps * bi != a.nbk - 1) {
      attn_fetch_block<T, D>(cx, p, layer, a, bi, f);
      f.done[bi] = true;
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <typename T, int D>
__device__ void attn_stage(Ctx& cx, const StepParams& p, int layer, AttnFetch<T, D>& f) {
  constexpr int KS = D / 16;            // k-steps over the head dimension
  constexpr int VROW = (D + 8) * 2;     // bytes of a staged V row (16 bytes of padding)
  constexpr int VBLK = 16 * VROW;       // one staged V block
  const int G = p.G, Hkv = p.Hkv;
  const int g = cx.lane >> 2, t = cx.lane & 3;
  const int total = cx.prefix[p.B];
  uint8_t* vst = cx.stage + cx.warp * 2 * VBLK;  // this warp's two staged V blocks
  T* out = reinterpret_cast<T*>(p.o);
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    const AttnUnit a = attn_unit(cx, p, u);
    const int b = a.b, h = a.h, c = a.c, L = a.L, nbk = a.nbk, nch = a.nch, jb = a.jb, nblk = a.nblk;
    float m_run = -INFINITY, l_run = 0.f;
    float oacc[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    if (nblk > 0) {
      // q rows of the group (heads h*G + g): lane (g, t) holds columns 16 ks + 4 t .. + 3
      uint2 qa[KS];
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks] = make_uint2(0u, 0u);
        if (g < G)
          qa[ks] = __ldcg(reinterpret_cast<const uint2*>(
              reinterpret_cast<const T*>(p.q) + static_cast<size_t>(b) * p.qd + (h * G + g) * D + 16 * ks + 4 * t));
      }
#pragma unroll
      for (int bi = 0; bi < 2; ++bi)
        if (bi < nblk && !(u == f.u && f.done[bi])) attn_fetch_block<T, D>(cx, p, layer, a, bi, f);
      cp_async_commit_wait_all();
      __syncwarp();
#pragma unroll
      for (int bi = 0; bi < 2; ++bi) {
        if (bi >= nblk) break;
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)
            SV<T>::mma(s[nt], qa[ks].x, 0u, qa[ks].y, 0u, f.kr[bi][ks][nt].x, f.kr[bi][ks][nt].y);
        }
        const int tok0 = (jb + kStepWarps * bi) * 16;
        float v[4];
        float mloc = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool valid = tok0 + nt * 8 + 2 * t + e < L;
            v[nt * 2 + e] = valid ? s[nt][e] * p.scale_log2 : -INFINITY;
            mloc = fmaxf(mloc, v[nt * 2 + e]);
          }
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
        const float m_new = fmaxf(m_run, mloc);
        const float alpha = exp2f(m_run - m_new);
        float pr[4], lsum = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pr[i] = exp2f(v[i] - m_new);
          lsum += pr[i];
        }
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
        l_run = l_run * alpha + lsum;
        m_run = m_new;
        // O^T columns are heads 2t, 2t + 1: their rescale factors live in quads 2t, 2t + 1
        const float a_e = __shfl_sync(0xffffffffu, alpha, (2 * t) * 4);
        const float a_o = __shfl_sync(0xffffffffu, alpha, (2 * t + 1) * 4);
        const uint32_t b0 = SV<T>::pack(pr[0], pr[1]);
        const uint32_t b1 = SV<T>::pack(pr[2], pr[3]);
        const uint32_t vb = smem_u32(vst + bi * VBLK) +
                            ((cx.lane & 7) + ((cx.lane >> 4) << 3)) * VROW + ((cx.lane >> 3) & 1) * 16;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          oacc[mt][0] *= a_e;
          oacc[mt][1] *= a_o;
          oacc[mt][2] *= a_e;
          oacc[mt][3] *= a_o;
          uint32_t am[4];
          ldsm_x4_trans(vb + mt * 32, am);
          SV<T>::mma(oacc[mt], am[0], am[1], am[2], am[3], b0, b1);
        }
      }
    }
    __syncwarp();
    // this warp's partial [G][D + 2] (accumulators, then m, l) over its own staged V
    float* wp = reinterpret_cast<float*>(vst);
    if (nblk > 0) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        if (2 * t < G) {
          wp[(2 * t) * (D + 2) + 16 * mt + g] = oacc[mt][0];
          wp[(2 * t) * (D + 2) + 16 * mt + g + 8] = oacc[mt][2];
        }
        if (2 * t + 1 < G) {
          wp[(2 * t + 1) * (D + 2) + 16 * mt + g] = oacc[mt][1];
          wp[(2 * t + 1) * (D + 2) + 16 * mt + g + 8] = oacc[mt][3];
        }
      }
      if (t == 0 && g < G) {
        wp[g * (D + 2) + D] = m_run;
        wp[g * (D + 2) + D + 1] = l_run;
      }
    }
    named_barrier_sync(1, kStepWarps * 32);
    // merge the warps in warp order
    const int nwv = min(kStepWarps, nbk - c * kStepAttnBlocks);
    float* part = p.attn_part + ((static_cast<size_t>(b) * Hkv + h) * p.max_ch) * G * (D + 2);
    for (int e = cx.tid; e < G * D; e += kStepWarps * 32) {
      const int hd = e / D, dim = e - hd * D;
      float M = -INFINITY;
      for (int w = 0; w < nwv; ++w)
        M = fmaxf(M, reinterpret_cast<const float*>(cx.stage + w * 2 * VBLK)[hd * (D + 2) + D]);
      float O = 0.f, Ls = 0.f;
      for (int w = 0; w < nwv; ++w) {
        const float* ww = reinterpret_cast<const float*>(cx.stage + w * 2 * VBLK) + hd * (D + 2);
        const float fw = exp2f(ww[D] - M);
        O += ww[dim] * fw;
        Ls += ww[D + 1] * fw;
      }
      if (nch == 1) {
        out[cm_index(b, (h * G + hd) * D + dim, p.B)] = SV<T>::from_f(O / Ls);
      } else {
        float* pc = part + (static_cast<size_t>(c) * G + hd) * (D + 2);
        pc[dim] = O;
        if (dim == 0) {
          pc[D] = M;
          pc[D + 1] = Ls;
        }
      }
    }
    if (nch > 1) {
      // the last unit of (row, head) to finish merges all of them in unit order
      __threadfence();
      named_barrier_sync(1, kStepWarps * 32);
      if (cx.tid == 0) {
        unsigned* cnt = p.sync + 2 + (static_cast<size_t>(layer) * kStepMaxRows + b) * Hkv + h;
        const unsigned old = atomicAdd(cnt, 1u);
        cx.ctl->flag = old + 1 == static_cast<unsigned>(nch);
      }
      named_barrier_sync(1, kStepWarps * 32);
      if (cx.ctl->flag) {
        __threadfence();
        // kE elements per thread and kMerge units per pass; a pass issues all its loads first
        constexpr int kE = 2, kMerge = 8;
        for (int e0 = cx.tid; e0 < G * D; e0 += kStepWarps * 32 * kE) {
          float mrun[kE], mprev[kE], orun[kE], lrun[kE];
#pragma unroll
          for (int r = 0; r < kE; ++r) mrun[r] = mprev[r] = -INFINITY, orun[r] = lrun[r] = 0.f;
          for (int c0 = 0; c0 < nch; c0 += kMerge) {
            float mv[kE][kMerge], ov[kE][kMerge], lv[kE][kMerge];
#pragma unroll
            for (int r = 0; r < kE; ++r) {
              const int e = e0 + r * kStepWarps * 32;
              const int hd = e / D, dim = e - hd * D;
#pragma unroll
              for (int u = 0; u < kMerge; ++u) {
                mv[r][u] = -INFINITY;
                ov[r][u] = lv[r][u] = 0.f;
                if (e < G * D && c0 + u < nch) {
                  const float* pc = part + (static_cast<size_t>(c0 + u) * G + hd) * (D + 2);
                  mv[r][u] = __ldcg(&pc[D]);
                  ov[r][u] = __ldcg(&pc[dim]);
                  lv[r][u] = __ldcg(&pc[D + 1]);
                }
              }
            }
#pragma unroll
            for (int r = 0; r < kE; ++r) {
              float M = -INFINITY;
#pragma unroll
              for (int u = 0; u < kMerge; ++u) M = fmaxf(M, mv[r][u]);
              mrun[r] = c0 == 0 ? M : fmaxf(mrun[r], M);
              // rescale what earlier passes summed to the running maximum
              const float f0 = c0 == 0 ? 0.f : exp2f(mprev[r] - mrun[r]);
              float O = orun[r] * f0, Ls = lrun[r] * f0;
#pragma unroll
              for (int u = 0; u < kMerge; ++u) {
                if (c0 + u < nch) {
                  const float fw = exp2f(mv[r][u] - mrun[r]);
                  O += ov[r][u] * fw;
                  Ls += lv[r][u] * fw;
                }
              }
              orun[r] = O;
              lrun[r] = Ls;
              mprev[r] = mrun[r];
            }
          }
#pragma unroll
          for (int r = 0; r < kE; ++r) {
            const int e = e0 + r * kStepWarps * 32;
            if (e < G * D) {
              const int hd = e / D, dim = e - hd * D;
              out[cm_index(b, (h * G + hd) * D + dim, p.B)] = SV<T>::from_f(orun[r] / lrun[r]);
            }
          }
        }
      }
    }
    named_barrier_sync(1, kStepWarps * 32);  // staged V, partials and flag are reused next
  }
}

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kStepThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  // ring | slot barriers | activation barrier | control | slots | scales | lengths | unit
  // offsets | split-K flags | RoPE table | activation slice | partial tiles (attention staging
  // over the last two)
  Ctx cx;
  cx.ring = smem;
  cx.full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.nslot) * kStepSlot);
  cx.empty = cx.full + p.nslot;
  cx.actbar = cx.empty + p.nslot;
  cx.ctl = reinterpret_cast<StepCtl*>(cx.actbar + 2);
  cx.s_slot = reinterpret_cast<long long*>(cx.ctl + 1);
  cx.rs = reinterpret_cast<float*>(cx.s_slot + kStepMaxRows);
  cx.s_seq = reinterpret_cast<int*>(cx.rs + kStepMaxRows);
  cx.prefix = cx.s_seq + kStepMaxRows;
  cx.last = cx.prefix + kStepMaxRows + 4;
  cx.s_cos = reinterpret_cast<float*>(cx.last + kStepMaxTilesPerCta);
  cx.s_sin = cx.s_cos + kStepMaxRows * (D / 2);
  cx.act = reinterpret_cast<uint8_t*>(cx.s_sin + kStepMaxRows * (D / 2));
  cx.red = reinterpret_cast<float*>(cx.act + kStepActBytes);
  cx.stage = cx.act;
  cx.actn = 0;
  cx.rows_valid = 0;
  cx.logits = nullptr;
  cx.warp = threadIdx.x >> 5;
  cx.lane = threadIdx.x & 31;
  cx.tid = threadIdx.x;
  cx.gen = 0;
  cx.seq = 0;
  cx.early_ok = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nslot; ++s) {
      mbar_init(&cx.full[s], 1);
      mbar_init(&cx.empty[s], kStepSlotChunks);  // every chunk of a slot is released once
    }
    mbar_init(cx.actbar, 1);
    cx.ctl->issued = 0;
    cx.ctl->abort = 0;
    cx.ctl->flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (cx.warp == kStepWarps) {
    // ------------------------------------------------------------ weight streaming warp
    if (cx.lane == 0) {
      const long long c0 = p.stream_off[blockIdx.x];
      const int n = static_cast<int>((p.with_lm ? p.stream_off[blockIdx.x + 1] : p.stream_lm[blockIdx.x]) - c0);
      const uint8_t* src = p.wpack + static_cast<size_t>(c0) * kStepChunk;
      const uint64_t pol = policy_evict_first();  // every weight byte is read once per step
      const int nb = (n + kStepSlotChunks - 1) / kStepSlotChunks;
      for (int j = 0; j < nb; ++j) {
        const int s = j % p.nslot;
        if (j >= p.nslot &&
            !mbar_wait(&cx.empty[s], static_cast<uint32_t>((j / p.nslot) - 1) & 1u, &cx.ctl->abort)) {
          if (!cta_aborted(cx)) {
            *reinterpret_cast<volatile int*>(&cx.ctl->abort) = 1;
            set_err(p.err, NS_DEV_WAIT_TIMEOUT);
          }
          break;
        }
        const int c1 = min(n, (j + 1) * kStepSlotChunks);
        const uint32_t bytes = static_cast<uint32_t>(c1 - j * kStepSlotChunks) * kStepChunk;
        mbar_arrive_expect_tx(&cx.full[s], bytes);
        bulk_g2s_hint(cx.ring + static_cast<size_t>(s) * kStepSlot,
                      src + static_cast<size_t>(j) * kStepSlot, bytes, &cx.full[s], pol);
        st_release_cta(&cx.ctl->issued, c1);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    step_setup<D>(cx, p);
    embed_stage<T>(cx, p);
    bool ok = grid_sync(cx, p);
    // projections in order: QKV, O, gate/up, down of every layer, then the LM head; attention
    // follows each QKV (one call site per stage function, so each is inlined once)
    const int n_proj = 4 * p.n_layers + (p.with_lm ? 1 : 0);
    for (int fi = 0; ok && fi < n_proj; ++fi) {
      const int l = fi >> 2, r = fi & 3;
      const int kind = l == p.n_layers ? SS_LM : r == 0 ? SS_QKV : r == 1 ? SS_O : r == 2 ? SS_GU : SS_DOWN;
      gemm_stage<T, D>(cx, p, kind, l);
      if (kind == SS_LM) break;
      if (kind == SS_QKV) {
        AttnFetch<T, D> af;
        attn_prepare<T, D>(cx, p, l, af);
        if (!grid_sync(cx, p)) break;
        attn_stage<T, D>(cx, p, l, af);
      }
      ok = grid_sync(cx, p);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  if (cx.ctl->abort && threadIdx.x == kStepWarps * 32) {
    // let this CTA's copies in flight land before its shared memory is released
    const int b_issued = (cx.ctl->issued + kStepSlotChunks - 1) / kStepSlotChunks;
    for (int j = max(0, b_issued - p.nslot); j < b_issued; ++j)
      (void)mbar_wait(&cx.full[j % p.nslot], static_cast<uint32_t>(j / p.nslot) & 1u, nullptr);
  }
}

// ------------------------------------------------------------------ weight packing
// One warp per chunk: lane (g, t) of pair half h2 of 32-column block kp holds, for rows g and
// g + 8 of the tile, columns 32 kp + 8 t + 4 h2 .. + 3 (the operand registers a0..a3 of
// mma.m16n8k16 under the column permutation described at the top of this file).
__global__ void step_pack_kernel(const PackDesc* desc, long long n, uint8_t* out, int head_dim) {
  const long long ci = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (ci >= n) return;
  const PackDesc ds = desc[ci];
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  auto row_of = [&](int r) -> long long {
    if (ds.kind == PK_ROPE) {
      const int dh = head_dim / 16, hh = ds.tile / dh, j = ds.tile - hh * dh;
      return static_cast<long long>(hh) * head_dim + (r < 8 ? j * 8 + r : head_dim / 2 + j * 8 + r - 8);
    }
    if (ds.kind == PK_GU) {
      // gate/up interleaved in 64-row groups [gate 64q .. 64q + 63 ; up 64q .. 64q + 63]
      const int f = ds.tile * 8 + (r & 7);
      return static_cast<long long>(f / 64) * 128 + (r < 8 ? 0 : 64) + f % 64;
    }
    return static_cast<long long>(ds.row0) + r;
  };
  const uint16_t* w = static_cast<const uint16_t*>(ds.w);
  const uint16_t* r0 = w + row_of(g) * ds.K;
  const uint16_t* r1 = w + row_of(g + 8) * ds.K;
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(ci) * kStepChunk);
#pragma unroll
  for (int kp = 0; kp < 4; ++kp)
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int k = ds.kc * 128 + kp * 32 + 8 * t + 4 * h2;
      uint4 v;
      v.x = *reinterpret_cast<const uint32_t*>(r0 + k);
      v.y = *reinterpret_cast<const uint32_t*>(r1 + k);
      v.z = *reinterpret_cast<const uint32_t*>(r0 + k + 2);
      v.w = *reinterpret_cast<const uint32_t*>(r1 + k + 2);
      dst[(kp * 2 + h2) * 32 + lane] = v;
    }
}

// ------------------------------------------------------------------ host side
size_t step_smem_bytes(int head_dim, int nslot) {
  const size_t red = static_cast<size_t>(kStepWarps) * kStepGroup * kStepMaxRows * kStepRedStride * 4;
  const size_t att = static_cast<size_t>(kStepWarps) * 2 * 16 * (head_dim + 8) * 2;
  const size_t uni = std::max(static_cast<size_t>(kStepActBytes) + red, att);
  return static_cast<size_t>(nslot) * (kStepSlot + 16) + 16 /* activation barrier */ + 16 /* control */ +
         8 * kStepMaxRows + 4 * kStepMaxRows + 4 * kStepMaxRows + 4 * (kStepMaxRows + 4) +
         4 * kStepMaxTilesPerCta + 2 * 4 * static_cast<size_t>(kStepMaxRows) * (head_dim / 2) + uni;
}

namespace {
template <typename T, int D>
cudaError_t configure_one(size_t smem, int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(step_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, step_kernel<T, D>, kStepThreads, smem);
}
}  // namespace

cudaError_t step_configure(int dtype, int head_dim, size_t smem, int* blocks_per_sm) {
  if (dtype == NS_BF16)
    return head_dim == 64 ? configure_one<__nv_bfloat16, 64>(smem, blocks_per_sm)
                          : configure_one<__nv_bfloat16, 128>(smem, blocks_per_sm);
  return head_dim == 64 ? configure_one<__half, 64>(smem, blocks_per_sm)
                        : configure_one<__half, 128>(smem, blocks_per_sm);
}

cudaError_t launch_step(const StepParams& p, int dtype, int grid, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kStepThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == NS_BF16)
    return p.d == 64 ? cudaLaunchKernelEx(&cfg, step_kernel<__nv_bfloat16, 64>, p)
                     : cudaLaunchKernelEx(&cfg, step_kernel<__nv_bfloat16, 128>, p);
  return p.d == 64 ? cudaLaunchKernelEx(&cfg, step_kernel<__half, 64>, p)
                   : cudaLaunchKernelEx(&cfg, step_kernel<__half, 128>, p);
}

bool build_step_plan(int grid, const StepParams& p, StepPlan* out) {
  out->stream_off.assign(grid + 1, 0);
  out->stream_lm.assign(grid, 0);
  for (int k = 0; k < SS_COUNT; ++k) {
    if (p.split[k] < 1 || p.split[k] > 8 || grid / p.split[k] < 1) return false;
    for (int c = 0; c < grid; ++c) {
      const StepTiles t = step_tiles(grid, c, p.n_tiles[k], p.kc[k], p.split[k], p.rot[k]);
      if (p.split[k] > 1 && t.count > kStepMaxTilesPerCta) return false;
    }
  }
  for (int c = 0; c < grid; ++c) {
    long long layer = 0;
    for (int k = 0; k < 4; ++k) {
      const StepTiles t = step_tiles(grid, c, p.n_tiles[k], p.kc[k], p.split[k], p.rot[k]);
      layer += static_cast<long long>(t.count) * (t.kc1 - t.kc0);
    }
    const StepTiles t = step_tiles(grid, c, p.n_tiles[SS_LM], p.kc[SS_LM], p.split[SS_LM], p.rot[SS_LM]);
    out->stream_lm[c] = out->stream_off[c] + layer * p.n_layers;
    out->stream_off[c + 1] = out->stream_lm[c] + static_cast<long long>(t.count) * (t.kc1 - t.kc0);
  }
  return true;
}

cudaError_t launch_step_pack(const PackDesc* desc, long long n, uint8_t* out, int head_dim,
                             cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const long long blocks = (n + 3) / 4;
  step_pack_kernel<<<static_cast<unsigned>(blocks), 128, 0, s>>>(desc, n, out, head_dim);
  return cudaGetLastError();
}

}  // namespace ns

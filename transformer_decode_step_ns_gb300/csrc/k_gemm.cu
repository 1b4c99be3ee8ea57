// Dense projections of the decode step on the 5th-generation tensor cores (tcgen05 / TMEM).
//
// "NanoFlow: LLM Serving Is Compute Bound ..." ("Four resource classes"): the KQV, O, Up/Gate
// and Down projections are the dense class -- compute bound once batched, weight-read bound at
// small batch ("The roofline flips": AI_decode ~ 2B).  One kernel serves both regimes:
//
//   D[128 features x BN tokens] = W_tile[128 x K] . X_tile[BN x K]^T   (UMMA M=128, N=BN)
//
// The weight is the UMMA "A" operand (so the batch is the N dimension, 16..256 tokens), both
// operands K-major, staged by TMA with 128-byte swizzle into an mbarrier ring; one thread
// issues tcgen05.mma into a TMEM accumulator; four warps read TMEM back for the epilogue.
// Split-K over CTAs (chosen from the weight's shape only, never from the batch) gives small
// matrices enough CTAs to stream HBM.  The split CTAs of a tile form one thread-block cluster
// and reduce through distributed shared memory in rank order (deterministic, no global
// workspace, no atomics); each cluster CTA then runs the fused epilogue for its share of tokens:
//   EPI_QKV    RMSNorm scale, RoPE on q/k, q store, k/v store into the paged cache slots
//              (nanoserve notes: RoPE once per step, slot mapping);
//   EPI_RESID  residual add, next RMSNorm's input x*gamma and per-tile sum of squares
//              (the "fused RMSNorm" of the nanoserve notes, folded into the producer);
//   EPI_SWIGLU silu(gate) * up on interleaved gate/up rows;
//   EPI_F32    fp32 output (LM head logits), optional RMSNorm scale.
// Weights are read before griddepcontrol.wait, so with programmatic dependent launch a GEMM
// streams its weights while the previous kernel of the step finishes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "ns_epi.cuh"
#include "ns_internal.h"
#include "ns_ptx.cuh"

namespace ns {

namespace {

template <typename T>
struct Cvt;
template <>
struct Cvt<__half> {
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ uint32_t bits(float x) { return __half_as_ushort(from_f(x)); }
};
template <>
struct Cvt<__nv_bfloat16> {
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) {
    return __float2bfloat16_rn(x);
  }
  static __device__ __forceinline__ uint32_t bits(float x) {
    return __bfloat16_as_ushort(from_f(x));
  }
};

// four values rounded to the storage type, in memory order, for one 8-byte store
template <typename T>
__device__ __forceinline__ uint2 pack4(float4 v) {
  return make_uint2(Cvt<T>::bits(v.x) | (Cvt<T>::bits(v.y) << 16),
                    Cvt<T>::bits(v.z) | (Cvt<T>::bits(v.w) << 16));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

constexpr uint32_t kABytes = kGemmTileN * kGemmTileK * 2;  // 16 KiB weight tile per stage
constexpr int kCtrlBytes = 2048;                            // barriers, flags, rs[256]

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kGemmThreads, 2)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int BN = p.BN;
  const uint32_t b_bytes = static_cast<uint32_t>(BN) * kGemmTileK * 2;
  const uint32_t stage_bytes = kABytes + b_bytes;
  uint8_t* ctrl = smem + static_cast<size_t>(p.nstage) * stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + p.nstage;
  uint64_t* accum = empty + p.nstage;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* last_flag = abort_flag + 1;
  int* issued = last_flag + 1;
  float* rs_s = reinterpret_cast<float*>(ctrl + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Token tiles vary fastest in launch order, so the CTAs that share a weight tile run
  // together and all but the first read it from L2.
  const int tile_m = blockIdx.x;
  const int split = blockIdx.y;
  const int tile_n = blockIdx.z;
  const int n0 = tile_n * kGemmTileN;
  const int nkb_total = p.K / kGemmTileK;
  const int kb0 = split * p.kb_per_split;
  const int nkb = min(p.kb_per_split, nkb_total - kb0);
  const int tok0 = p.row0 + tile_m * BN;
  const int m_valid = min(BN, p.M - tile_m * BN);
  const uint32_t ncols = BN <= 32 ? 32u : BN <= 64 ? 64u : BN <= 128 ? 128u : 256u;

  auto stageA = [&](int s) { return smem + static_cast<size_t>(s) * stage_bytes; };
  auto stageB = [&](int s) { return smem + static_cast<size_t>(s) * stage_bytes + kABytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    *abort_flag = 0;
    *last_flag = 0;
    *issued = 0;
    fence_mbar_init();
    prefetch_tmap(&mapA);
    prefetch_tmap(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int S = p.splits;
  const int rank = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int n_own = m_valid > rank ? (m_valid - rank + S - 1) / S : 0;  // owned tokens
  const bool two_pass = gemm_two_pass(BN);
  // the QKV epilogue stages its q/k columns' RoPE rows in the ring when they fit behind the tile
  const bool qkv_staged =
      p.epi == EPI_QKV && !two_pass && n0 < p.e.q_dim + p.e.kv_dim &&
      static_cast<size_t>(n_own) * 8 * (p.e.head_dim >> 1) + static_cast<size_t>(BN) * kGemmTileN * 4 <=
          static_cast<size_t>(p.nstage) * stage_bytes;
  // the residual epilogue stages the old residual rows of its owned tokens the same way
  const size_t tile_bytes = static_cast<size_t>(two_pass ? kPassRows : BN) * kGemmTileN * 4;
  const bool resid_staged =
      p.epi == EPI_RESID && static_cast<size_t>(n_own) * kGemmTileN * 4 + tile_bytes <=
                                static_cast<size_t>(p.nstage) * stage_bytes;
  // the residual epilogue's next-norm gains for the lane's four features (loaded early)
  float4 gam4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const uint32_t tmem = *tmem_slot;
  // Dependents may be scheduled once every CTA holds its TMEM (so none of them can starve us).
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && nkb > 0) {
      // a weight tile read by one CTA only is streamed; one shared by several token tiles stays
      const uint64_t pol_w = gridDim.x > 1 ? policy_evict_normal() : policy_evict_first();
      const int pre = min(p.nstage, nkb);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], stage_bytes);
        tma_load_2d_hint(stageA(i), &mapA, &full[i], (kb0 + i) * kGemmTileK, n0, pol_w);
      }
      griddep_wait();  // activations come from the previous kernel of the step
      for (int i = 0; i < pre; ++i) tma_load_2d(stageB(i), &mapB, &full[i], (kb0 + i) * kGemmTileK, tok0);
      int i = pre;
      for (; i < nkb; ++i) {
        const int s = i % p.nstage;
        const uint32_t ph = static_cast<uint32_t>((i / p.nstage) - 1) & 1u;
        if (!mbar_wait(&empty[s], ph, abort_flag)) {
          *abort_flag = 1;
          set_err(p.err, NS_DEV_WAIT_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        tma_load_2d_hint(stageA(s), &mapA, &full[s], (kb0 + i) * kGemmTileK, n0, pol_w);
        tma_load_2d(stageB(s), &mapB, &full[s], (kb0 + i) * kGemmTileK, tok0);
      }
      *issued = i;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nkb; ++i) {
        const int s = i % p.nstage;
        if (!mbar_wait(&full[s], static_cast<uint32_t>(i / p.nstage) & 1u, abort_flag)) {
          *abort_flag = 1;
          set_err(p.err, NS_DEV_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(stageA(s));
        const uint32_t b_addr = smem_u32(stageB(s));
#pragma unroll
        for (int k = 0; k < kGemmTileK / 16; ++k) {
          umma_f16(tmem, sw128_kmajor_desc(a_addr + k * 32), sw128_kmajor_desc(b_addr + k * 32),
                   p.idesc, (i | k) != 0 ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(accum);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue warps
    // What the epilogue reads besides the accumulator is loaded while the main loop runs (the
    // RMSNorm scale of each owned token, the next norm's gains) or copied into the ring as soon
    // as the accumulator is complete (the QKV epilogue's RoPE rows, the residual epilogue's old
    // residual rows), where it lands during the TMEM read-out and the split-K reduction.
    const EpiArgs& e = p.e;
    const int et = threadIdx.x - 64;  // 0..127
    const int ew = warp - 2;
    // inputs fixed before the step starts (metadata, weights)
    if (p.epi == EPI_RESID) gam4 = *reinterpret_cast<const float4*>(e.gamma_next + n0 + 4 * lane);
    griddep_wait();  // the previous kernel wrote the rest and may still read our outputs
    if (e.sumsq_in != nullptr) {
      // rs[j] = rsqrt(sum of the row's per-tile partial sums / H + eps): one warp per token,
      // lanes over the partials, a fixed shuffle tree (the order depends on H only)
      const int n_tiles = e.sumsq_tiles;
      const size_t ld = static_cast<size_t>(e.sumsq_ld);
      for (int jj0 = ew; jj0 < n_own; jj0 += 16) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jj = jj0 + 4 * u;
          const float* sp = e.sumsq_in + tok0 + rank + S * jj;
          v[u] = 0.f;
          if (jj < n_own) {
            if (n_tiles <= 64) {
              const float x0 = lane < n_tiles ? sp[lane * ld] : 0.f;
              const float x1 = lane + 32 < n_tiles ? sp[(lane + 32) * ld] : 0.f;
              v[u] = x0 + x1;
            } else {
              for (int t = lane; t < n_tiles; t += 32) v[u] += sp[t * ld];
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float x = v[u];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
          const int jj = jj0 + 4 * u;
          if (lane == 0 && jj < n_own) rs_s[rank + S * jj] = rms_scale(x, e.norm_dim, e.eps);
        }
      }
    }
    // TMEM -> shared tile [BN][128] fp32 (reuses the stage ring: every MMA has completed)
    const int q = warp & 3;             // TMEM lane quarter this warp may read
    const int row = q * 32 + lane;      // output feature within the tile
    const bool ok = mbar_wait(accum, 0, abort_flag);
    tc_fence_after();
    if (!ok) {
      *abort_flag = 1;
      set_err(p.err, NS_DEV_WAIT_TIMEOUT);
    }
    float* tile = reinterpret_cast<float*>(smem);
    // The RoPE cos/sin rows of the owned tokens go into the ring behind the staged tile (every
    // MMA has completed, so the ring is free); they land while the tile is read out of TMEM and
    // reduced across the cluster.  [owned token][cos half | sin half] fp32.
    if (ok && !*abort_flag && resid_staged) {
      const uint32_t base = smem_u32(smem) + static_cast<uint32_t>(tile_bytes);
      for (int idx = et; idx < n_own * (kGemmTileN / 4); idx += 128) {
        const int k = idx >> 5, pc = idx & 31;
        cp_async_16(base + static_cast<uint32_t>((k * kGemmTileN + 4 * pc) * 4),
                    e.resid + static_cast<size_t>(tok0 + rank + S * k) * e.resid_dim + n0 + 4 * pc);
      }
    }
    if (ok && !*abort_flag && qkv_staged) {
      const int half = e.head_dim >> 1, pieces = half >> 1;  // 16-byte pieces per token
      const uint32_t base = smem_u32(smem) + static_cast<uint32_t>(BN) * kGemmTileN * 4;
      for (int idx = et; idx < n_own * pieces; idx += 128) {
        const int k = idx / pieces, pc = idx - k * pieces;
        const bool is_cos = pc < (pieces >> 1);
        const float* src = (is_cos ? e.rope_cos : e.rope_sin) +
                           static_cast<size_t>(tok0 + rank + S * k) * half +
                           4 * (is_cos ? pc : pc - (pieces >> 1));
        cp_async_16(base + static_cast<uint32_t>((k * 2 * half + 4 * pc) * 4), src);
      }
    }
    const int nchunk = (m_valid + 15) >> 4;
    if (ok && !*abort_flag && !two_pass) {
      for (int c = 0; c < nchunk; ++c) {
        uint32_t r[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c * 16), r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) tile[(c * 16 + i) * kGemmTileN + row] = __uint_as_float(r[i]);
      }
    }
  }

  // ------------------------------------------------------------------ split-K reduction
  // The split CTAs of one output tile form a thread-block cluster.  CTA `rank` owns tokens
  // j = rank, rank + S, ...; it sums their partial rows over every CTA of the cluster through
  // distributed shared memory, in rank order (deterministic), then runs the epilogue for them.
  // Cluster barrier phases, per staged pass: "every tile is complete" before the reduction and
  // "every peer has finished reading" before the tile is overwritten or the CTA leaves; the
  // second is arrived at as soon as a thread is done with remote reads and waited for late.
  // A tile wider than kPassRows tokens is staged kPassRows tokens at a time (its shared-memory
  // tile is then half the size, so two CTAs fit on an SM).
  const int npass = two_pass ? (m_valid + kPassRows - 1) / kPassRows : 1;
  __syncthreads();
  if (S > 1 && !two_pass) {
    cluster_sync();
    if (warp < 2) cluster_arrive();  // these warps read no peer memory
  }
  if (S > 1 && two_pass && warp < 2) {
    for (int pass = 0; pass < npass; ++pass) {  // the same phases as the epilogue warps
      if (pass > 0) cluster_wait();
      cluster_sync();
      cluster_arrive();
    }
  }
  if (warp >= 2) {
    const int et = threadIdx.x - 64;  // 0..127: feature within the tile
    const int ew = warp - 2;
    const bool run = !*abort_flag;
    float* const tbase = reinterpret_cast<float*>(smem);
    // owned tokens j = rank + S * k with lo <= j < hi (rows j - lo of the staged tile)
    auto reduce = [&](int k_lo, int k_hi, int lo) {
      // thread -> 4 consecutive features of every 4th owned token; all ranks' float4 loads
      // are issued before they are summed (in rank order)
      const uint32_t base = smem_u32(tbase);
      const int fg = et & 31, slot = et >> 5;
      for (int k = k_lo + slot; k < k_hi; k += 4) {
        const int row = rank + S * k - lo;
        const uint32_t off = base + static_cast<uint32_t>((row * kGemmTileN + 4 * fg) * 4);
        float4 v[kMaxSplits];
#pragma unroll
        for (int r = 0; r < kMaxSplits; ++r)
          if (r < S) v[r] = ld_shared_cluster_f32x4(map_shared_rank(off, r));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kMaxSplits; ++r) {
          if (r < S) {
            acc.x += v[r].x;
            acc.y += v[r].y;
            acc.z += v[r].z;
            acc.w += v[r].w;
          }
        }
        *reinterpret_cast<float4*>(&tbase[row * kGemmTileN + 4 * fg]) = acc;
      }
    };
    if (!two_pass) {
      if (run && S > 1) reduce(0, n_own, 0);
      if (qkv_staged || resid_staged) cp_async_commit_wait_all();  // this thread's rows landed
      named_barrier_sync(1, 128);  // reduced rows, RMSNorm scales and RoPE rows are in shared memory
      if (S > 1) cluster_arrive();  // this CTA's remote reads are complete
    }
    const EpiArgs& e = p.e;
    const bool scaled = e.sumsq_in != nullptr;
    for (int pass = 0; pass < npass; ++pass) {
      // token rows [lo, hi) of the CTA's tile; owned tokens k_lo <= k < k_hi among them
      const int lo = two_pass ? pass * kPassRows : 0;
      const int hi = two_pass ? min(lo + kPassRows, m_valid) : m_valid;
      const int k_lo = two_pass ? max(0, (lo - rank + S - 1) / S) : 0;
      const int k_hi = two_pass ? max(k_lo, (hi - rank + S - 1) / S) : n_own;
      const int jn = k_hi - k_lo;
      if (two_pass) {
        if (pass > 0) {
          named_barrier_sync(1, 128);  // this CTA is done with the previous pass's tile
          if (S > 1) cluster_wait();   // ... and so are its peers
        }
        const int q = warp & 3, frow = q * 32 + lane;
        if (run) {
          for (int c = 0; c < (hi - lo + 15) >> 4; ++c) {
            uint32_t r[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(lo + c * 16), r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) tbase[(c * 16 + i) * kGemmTileN + frow] = __uint_as_float(r[i]);
          }
        }
        if (resid_staged && pass == 0) cp_async_commit_wait_all();  // this thread's rows landed
        named_barrier_sync(1, 128);
        if (S > 1) {
          cluster_sync();
          if (run) reduce(k_lo, k_hi, lo);
          named_barrier_sync(1, 128);
          cluster_arrive();
        }
      }
      if (run) {
        // tile[j * 128 + r] addresses the staged row of token j of this pass
        float* tile = tbase - static_cast<ptrdiff_t>(lo) * kGemmTileN;
        auto tok_of = [&](int k) { return rank + S * (k_lo + k); };  // k-th owned token of the pass
        if (p.epi == EPI_F32) {
          float* out = e.out_f32;
          if (e.out_ptr_slot != nullptr) out = reinterpret_cast<float*>(*e.out_ptr_slot);
          // padding rows of a bucketed graph have no output row
          const int n_rows = e.rows_valid != nullptr ? *e.rows_valid - tok0 : m_valid;
          for (int idx = et; idx < jn * kGemmTileN; idx += 128) {
            const int j = tok_of(idx >> 7), r = idx & 127;
            if (j >= n_rows) continue;
            float v = tile[j * kGemmTileN + r];
            if (scaled) v *= rs_s[j];
            out[static_cast<size_t>(tok0 + j) * e.ldo + n0 + r] = v;
          }
        } else if (p.epi == EPI_QKV) {
          // A warp takes whole owned tokens (the pass's k = ew, ew + 4, ...); lane l holds
          // features 4l .. 4l + 3 of the tile.  The RoPE partners (i, i + d/2) of a head sit
          // half/4 lanes apart and swap values by shuffles; a token costs one 16-byte read of
          // the tile, of cos and of sin, one 8-byte store, and one cache address per lane.
          // Each element gets the formulas of the persistent kernel's epilogue.
          const int d = e.head_dim, half = d >> 1;
          const bool is_q = n0 < e.q_dim;
          const bool is_k = !is_q && n0 < e.q_dim + e.kv_dim;
          const bool rope = is_q || is_k;
          const int f0 = 4 * lane;
          const int fd = f0 % d;  // feature within its head
          const bool low = fd < half;
          const int i0 = low ? fd : fd - half;  // RoPE pair of the lane's first feature
          const int plane = half >> 2;          // lanes between partners
          const int col = n0 - e.q_dim - (is_k || is_q ? 0 : e.kv_dim) + f0;  // within K or V
          const int kvh = col / d, dim = col - kvh * d;
          const float* staged = reinterpret_cast<const float*>(smem + static_cast<size_t>(BN) * kGemmTileN * 4);
          for (int kk0 = ew; kk0 < jn; kk0 += 128) {
            // lane t holds the cache slot of the warp's token kk0 + 4t
            long long my_slot = 0;
            if (!is_q && kk0 + 4 * lane < jn) my_slot = e.slot_mapping[tok0 + tok_of(kk0 + 4 * lane)];
            const int nt = min(32, (jn - kk0 + 3) >> 2);  // the warp's tokens in this batch
#pragma unroll 2
            for (int t = 0; t < nt; ++t) {
              const int kk = kk0 + 4 * t;
              const int j = tok_of(kk), tok = tok0 + j;
              float4 x = *reinterpret_cast<const float4*>(&tile[j * kGemmTileN + f0]);
              if (scaled) {
                const float sc = rs_s[j];
                x.x *= sc;
                x.y *= sc;
                x.z *= sc;
                x.w *= sc;
              }
              if (rope) {
                float4 c, sn;
                if (qkv_staged) {
                  const float* row = staged + static_cast<size_t>(k_lo + kk) * 2 * half;
                  c = *reinterpret_cast<const float4*>(row + i0);
                  sn = *reinterpret_cast<const float4*>(row + half + i0);
                } else {
                  const size_t o = static_cast<size_t>(tok) * half + i0;
                  c = *reinterpret_cast<const float4*>(e.rope_cos + o);
                  sn = *reinterpret_cast<const float4*>(e.rope_sin + o);
                }
                const float4 xp = make_float4(__shfl_xor_sync(0xffffffffu, x.x, plane),
                                              __shfl_xor_sync(0xffffffffu, x.y, plane),
                                              __shfl_xor_sync(0xffffffffu, x.z, plane),
                                              __shfl_xor_sync(0xffffffffu, x.w, plane));
                if (low) {
                  x = make_float4(rope_lo(x.x, xp.x, c.x, sn.x), rope_lo(x.y, xp.y, c.y, sn.y),
                                  rope_lo(x.z, xp.z, c.z, sn.z), rope_lo(x.w, xp.w, c.w, sn.w));
                } else {
                  x = make_float4(rope_hi(xp.x, x.x, c.x, sn.x), rope_hi(xp.y, x.y, c.y, sn.y),
                                  rope_hi(xp.z, x.z, c.z, sn.z), rope_hi(xp.w, x.w, c.w, sn.w));
                }
              }
              const uint2 v4 = pack4<T>(x);
              if (is_q) {
                *reinterpret_cast<uint2*>(reinterpret_cast<T*>(e.q_out) +
                                          static_cast<size_t>(tok) * e.q_dim + n0 + f0) = v4;
              } else {
                const long long slot = __shfl_sync(0xffffffffu, my_slot, t);
                if (slot < 0 || slot >= e.pool_slots) {
                  if (lane == 0) set_err(p.err, NS_DEV_BAD_SLOT);
                  continue;
                }
                T* pool = reinterpret_cast<T*>(is_k ? e.k_pool : e.v_pool);
                const size_t base = ((static_cast<size_t>(slot / e.block_size) * e.n_kv_heads + kvh) *
                                         e.block_size + static_cast<size_t>(slot % e.block_size)) * d;
                *reinterpret_cast<uint2*>(pool + base + dim) = v4;
                if (e.kv_stage != nullptr)
                  *reinterpret_cast<uint2*>(reinterpret_cast<T*>(e.kv_stage) +
                                            static_cast<size_t>(tok) * 2 * e.kv_dim +
                                            (is_k ? 0 : e.kv_dim) + col) = v4;
              }
            }
          }
          // q and the cache are read by ordinary loads and cp.async (no async-proxy fence)
        } else if (p.epi == EPI_RESID) {
          // A warp takes whole owned tokens; lane l holds features 4l .. 4l + 3: the new
          // residual, the next norm's input and the square that the per-token sum below reads.
          T* xo = reinterpret_cast<T*>(e.xn_out);
          const int f0 = 4 * lane;
          const float* staged = reinterpret_cast<const float*>(smem + tile_bytes);
#pragma unroll 4
          for (int kk = ew; kk < jn; kk += 4) {
            const int j = tok_of(kk);
            const size_t gi = static_cast<size_t>(tok0 + j) * e.resid_dim + n0 + f0;
            float4* tp = reinterpret_cast<float4*>(&tile[j * kGemmTileN + f0]);
            const float4 x = *tp;
            const float4 old =
                resid_staged ? *reinterpret_cast<const float4*>(staged + static_cast<size_t>(k_lo + kk) * kGemmTileN + f0)
                             : *reinterpret_cast<const float4*>(e.resid + gi);
            const float4 rn = make_float4(old.x + x.x, old.y + x.y, old.z + x.z, old.w + x.w);
            *reinterpret_cast<float4*>(e.resid + gi) = rn;
            *reinterpret_cast<uint2*>(xo + gi) =
                pack4<T>(make_float4(rn.x * gam4.x, rn.y * gam4.y, rn.z * gam4.z, rn.w * gam4.w));
            *tp = make_float4(rn.x * rn.x, rn.y * rn.y, rn.z * rn.z, rn.w * rn.w);
          }
          named_barrier_sync(1, 128);
          for (int k = ew; k < jn; k += 4) {
            const int j = tok_of(k);
            const float* tr = tile + j * kGemmTileN;
            float s = (tr[lane] + tr[lane + 32]) + (tr[lane + 64] + tr[lane + 96]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) e.sumsq_out[static_cast<size_t>(tile_n) * e.sumsq_ld + tok0 + j] = s;
          }
          fence_proxy_async_global();
        } else if (p.epi == EPI_SWIGLU) {
          // a warp takes whole owned tokens; lane l makes outputs 2l and 2l + 1 of the tile's 64
          // (gate rows 0-63, up rows 64-127)
          T* ao = reinterpret_cast<T*>(e.act_out);
          const int f0 = tile_n * 64;
#pragma unroll 4
          for (int kk = ew; kk < jn; kk += 4) {
            const int j = tok_of(kk);
            const float sc = scaled ? rs_s[j] : 1.f;
            const float2 g = *reinterpret_cast<const float2*>(&tile[j * kGemmTileN + 2 * lane]);
            const float2 u = *reinterpret_cast<const float2*>(&tile[j * kGemmTileN + 64 + 2 * lane]);
            const float a0 = silu_mul(g.x * sc, u.x * sc), a1 = silu_mul(g.y * sc, u.y * sc);
            *reinterpret_cast<uint32_t*>(ao + static_cast<size_t>(tok0 + j) * e.ffn + f0 + 2 * lane) =
                Cvt<T>::bits(a0) | (Cvt<T>::bits(a1) << 16);
          }
          fence_proxy_async_global();
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  // no CTA of the cluster may leave while a peer still reads its tile
  if (S > 1) cluster_wait();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // Let this CTA's own copies in flight land before its shared memory is released.
    const int n_issued = *issued;
    for (int i = max(0, n_issued - p.nstage); i < n_issued; ++i) {
      (void)mbar_wait(&full[i % p.nstage], static_cast<uint32_t>(i / p.nstage) & 1u, nullptr);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ------------------------------------------------------------------------------ persistent
// Long launches of an unsplit weight (more than 64 rows at the ridge point and in the
// compute-bound dense batches of the NanoFlow page, and vocabulary-wide heads at any row count)
// run a persistent variant: one CTA per SM loops over
// work units (token tile, 128-feature tile), token tiles fastest so CTAs running side by side
// share a weight tile through L2.  The TMA warp streams every unit's stages through one deep
// ring without stopping between units; the MMA warp alternates between two TMEM accumulators,
// so the epilogue of one unit overlaps the main loop of the next.  The epilogue runs from
// registers (a thread holds one feature of 16 tokens; RoPE pairs, gate/up pairs and the
// per-token sums of squares are exchanged through a 16-token shared buffer) with the cluster
// kernel's formulas and summation orders, so a row gets the same bits from either kernel.
// Nothing waits on another CTA, so any grid size is safe.
constexpr int kXchgFloats = 16 * kGemmTileN;  // one 16-token chunk of a tile

template <typename T>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_persistent_kernel(const __grid_constant__ CUtensorMap mapA,
                           const __grid_constant__ CUtensorMap mapB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int BN = p.BN;
  const int ns = p.nstage;
  const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(BN) * kGemmTileK * 2;
  float* xchg = reinterpret_cast<float*>(smem + static_cast<size_t>(ns) * stage_bytes);
  uint8_t* ctrl = reinterpret_cast<uint8_t*>(xchg + kXchgFloats);
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + ns;
  uint64_t* acc_full = empty + ns;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* issued = abort_flag + 1;
  int* epi_flag = issued + 1;  // broadcast word of the epilogue warps
  float* rs_s = reinterpret_cast<float*>(ctrl + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = p.tiles_m, n_tiles = p.N / kGemmTileN;
  const int n_units = tiles_m * n_tiles;
  const int nkb_total = p.K / kGemmTileK;
  const uint32_t ncols = BN <= 128 ? 128u : 256u;

  auto stageA = [&](int st) { return smem + static_cast<size_t>(st) * stage_bytes; };
  auto stageB = [&](int st) { return smem + static_cast<size_t>(st) * stage_bytes + kABytes; };
  // unit u -> (token tile, feature tile); every unit runs all k-blocks
  struct Unit {
    int tm, tn, kb0, nkb;
  };
  auto unit_of = [&](int u) {
    Unit w;
    w.tm = u % tiles_m;
    w.tn = u / tiles_m;
    w.kb0 = 0;
    w.nkb = nkb_total;
    return w;
  };

  if (threadIdx.x == 0) {
    for (int st = 0; st < ns; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    *abort_flag = 0;
    *issued = 0;
    fence_mbar_init();
    prefetch_tmap(&mapA);
    prefetch_tmap(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = tiles_m > 1 ? policy_evict_normal() : policy_evict_first();
      // (unit, k-block) pairs of this CTA in order; `it` counts them
      int u = blockIdx.x, i = 0, it = 0;
      Unit w = u < n_units ? unit_of(u) : Unit{};
      auto next = [&]() {
        if (++i == w.nkb) {
          i = 0;
          u += gridDim.x;
          if (u < n_units) w = unit_of(u);
        }
      };
      // the weights of the first ring's worth of stages go out before the dependency wait
      const int u0 = u;
      const Unit w0 = w;
      int pre = 0;
      while (pre < ns && u < n_units) {
        mbar_arrive_expect_tx(&full[pre], stage_bytes);
        tma_load_2d_hint(stageA(pre), &mapA, &full[pre], (w.kb0 + i) * kGemmTileK, w.tn * kGemmTileN, pol_w);
        ++pre;
        next();
      }
      griddep_wait();  // activations come from the previous kernel of the step
      {
        int uu = u0, ii = 0;
        Unit ww = w0;
        for (int t = 0; t < pre; ++t) {
          tma_load_2d(stageB(t), &mapB, &full[t], (ww.kb0 + ii) * kGemmTileK, p.row0 + ww.tm * BN);
          if (++ii == ww.nkb) {
            ii = 0;
            uu += gridDim.x;
            if (uu < n_units) ww = unit_of(uu);
          }
        }
      }
      it = pre;
      while (u < n_units) {
        const int st = it % ns;
        if (!mbar_wait(&empty[st], static_cast<uint32_t>((it / ns) - 1) & 1u, abort_flag)) {
          *abort_flag = 1;
          set_err(p.err, NS_DEV_WAIT_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[st], stage_bytes);
        tma_load_2d_hint(stageA(st), &mapA, &full[st], (w.kb0 + i) * kGemmTileK, w.tn * kGemmTileN, pol_w);
        tma_load_2d(stageB(st), &mapB, &full[st], (w.kb0 + i) * kGemmTileK, p.row0 + w.tm * BN);
        ++it;
        next();
      }
      *issued = it;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, j = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
        const Unit w = unit_of(u);
        const int b = j & 1;
        if (j >= 2 && !mbar_wait(&acc_empty[b], static_cast<uint32_t>((j >> 1) - 1) & 1u, abort_flag)) {
          *abort_flag = 1;
          set_err(p.err, NS_DEV_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b) * ncols;
        bool ok = true;
        for (int i = 0; i < w.nkb; ++i, ++it) {
          const int st = it % ns;
          if (!mbar_wait(&full[st], static_cast<uint32_t>(it / ns) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stageA(st));
          const uint32_t b_addr = smem_u32(stageB(st));
#pragma unroll
          for (int k = 0; k < kGemmTileK / 16; ++k) {
            umma_f16(d, sw128_kmajor_desc(a_addr + k * 32), sw128_kmajor_desc(b_addr + k * 32), p.idesc,
                     (i | k) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[st]);
        }
        if (!ok) {
          *abort_flag = 1;
          set_err(p.err, NS_DEV_WAIT_TIMEOUT);
          break;
        }
        umma_commit(&acc_full[b]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue warps
    const EpiArgs& e = p.e;
    const int et = threadIdx.x - 64;  // 0..127
    const int ew = warp - 2;
    const int q = warp & 3;           // TMEM lane quarter this warp may read
    const int f = q * 32 + lane;      // output feature within the tile
    const bool scaled = e.sumsq_in != nullptr;
    griddep_wait();  // the previous kernel wrote the epilogue's inputs and may read our outputs
    int j = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
      const Unit w = unit_of(u);
      const int b = j & 1;
      const int n0 = w.tn * kGemmTileN;
      const int tok0 = p.row0 + w.tm * BN;
      const int m_valid = min(BN, p.M - w.tm * BN);
      const int nchunk = (m_valid + 15) >> 4;
      if (scaled) {
        // rs[j] = rsqrt(sum of the row's per-tile partial sums / H + eps) for the unit's tokens,
        // while the main loop runs.  One thread per token with all its loads in flight; the sum
        // follows the cluster kernel's shuffle tree exactly: lane l first adds partials
        // l, l + 32, l + 64, ... in order, then the xor tree halves the lanes (lane l + o into
        // lane l for o = 16, 8, 4, 2, 1), so the result is bitwise the same.
        const int n_tiles_s = e.sumsq_tiles;
        const size_t ld = static_cast<size_t>(e.sumsq_ld);
        for (int jj = et; jj < m_valid; jj += 128) {
          const float* sp = e.sumsq_in + tok0 + jj;
          float x[32];
          if (n_tiles_s <= 64) {
            float x0[32], x1[32];
#pragma unroll
            for (int l = 0; l < 32; ++l) {
              x0[l] = l < n_tiles_s ? sp[l * ld] : 0.f;
              x1[l] = l + 32 < n_tiles_s ? sp[(l + 32) * ld] : 0.f;
            }
#pragma unroll
            for (int l = 0; l < 32; ++l) x[l] = x0[l] + x1[l];
          } else {
#pragma unroll
            for (int l = 0; l < 32; ++l) {
              x[l] = 0.f;
              for (int t = l; t < n_tiles_s; t += 32) x[l] += sp[t * ld];
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int l = 0; l < o; ++l) x[l] = x[l] + x[l + o];
          }
          rs_s[jj] = rms_scale(x[0], e.norm_dim, e.eps);
        }
      }
      // one thread waits for the accumulator (bounded) and tells the others; the barrier also
      // publishes rs
      if (et == 0) {
        const bool ok = !*abort_flag && mbar_wait(&acc_full[b], static_cast<uint32_t>(j >> 1) & 1u, abort_flag);
        if (!ok) {
          *abort_flag = 1;
          set_err(p.err, NS_DEV_WAIT_TIMEOUT);
        }
        *epi_flag = ok ? 1 : 0;
      }
      named_barrier_sync(1, 128);
      if (!*epi_flag) break;
      tc_fence_after();
      const uint32_t tb = tmem + static_cast<uint32_t>(b) * ncols + (static_cast<uint32_t>(q * 32) << 16);
      {
        const int d = e.head_dim, half = d >> 1;
        const bool qk_tile = p.epi == EPI_QKV && n0 < e.q_dim + e.kv_dim;
        for (int c = 0; c < nchunk; ++c) {
          float v[16];
          {
            uint32_t r[16];
            tmem_ld16(tb + static_cast<uint32_t>(c * 16), r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
          }
          if (p.epi == EPI_F32) {
            float* out = e.out_f32;
            if (e.out_ptr_slot != nullptr) out = reinterpret_cast<float*>(*e.out_ptr_slot);
            const int n_rows = e.rows_valid != nullptr ? min(m_valid, *e.rows_valid - tok0) : m_valid;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jj = c * 16 + i;
              if (jj >= n_rows) continue;
              float val = v[i];
              if (scaled) val *= rs_s[jj];
              out[static_cast<size_t>(tok0 + jj) * e.ldo + n0 + f] = val;
            }
          } else if (p.epi == EPI_RESID) {
            T* xo = reinterpret_cast<T*>(e.xn_out);
            const float gam = e.gamma_next[n0 + f];
            float old[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jj = c * 16 + i;
              old[i] = jj < m_valid ? e.resid[static_cast<size_t>(tok0 + jj) * e.resid_dim + n0 + f] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jj = c * 16 + i;
              float sq = 0.f;
              if (jj < m_valid) {
                const size_t gi = static_cast<size_t>(tok0 + jj) * e.resid_dim + n0 + f;
                const float rn = old[i] + v[i];
                e.resid[gi] = rn;
                xo[gi] = Cvt<T>::from_f(rn * gam);
                sq = rn * rn;
              }
              xchg[i * kGemmTileN + f] = sq;
            }
            named_barrier_sync(1, 128);
            for (int i = ew; i < 16; i += 4) {
              const int jj = c * 16 + i;
              const float* tr = xchg + i * kGemmTileN;
              float sm = (tr[lane] + tr[lane + 32]) + (tr[lane + 64] + tr[lane + 96]);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
              if (lane == 0 && jj < m_valid) e.sumsq_out[static_cast<size_t>(w.tn) * e.sumsq_ld + tok0 + jj] = sm;
            }
            named_barrier_sync(1, 128);
          } else if (p.epi == EPI_SWIGLU) {
            T* ao = reinterpret_cast<T*>(e.act_out);
            if (q >= 2) {
#pragma unroll
              for (int i = 0; i < 16; ++i) xchg[i * kGemmTileN + f] = v[i];  // up rows
            }
            named_barrier_sync(1, 128);
            if (q < 2) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int jj = c * 16 + i;
                if (jj >= m_valid) continue;
                const float sc = scaled ? rs_s[jj] : 1.f;
                const float g = v[i] * sc;
                const float up = xchg[i * kGemmTileN + 64 + f] * sc;
                ao[static_cast<size_t>(tok0 + jj) * e.ffn + w.tn * 64 + f] = Cvt<T>::from_f(silu_mul(g, up));
              }
            }
            named_barrier_sync(1, 128);
          } else if (qk_tile) {
            // q and k columns: RoPE pairs (i, i + d/2) of each head, partners exchanged
            T* qo = reinterpret_cast<T*>(e.q_out);
            T* kp = reinterpret_cast<T*>(e.k_pool);
            const int hf = f % d, ip = hf % half;
            const bool lo = hf < half;
            const int partner = lo ? f + half : f - half;
            const bool k_tile = n0 >= e.q_dim;
            // this chunk's angles and slots, loaded before anything is stored
            float csv[16], snv[16];
            long long slv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jj = c * 16 + i;
              const int tok = tok0 + min(jj, m_valid - 1);
              const size_t o = static_cast<size_t>(tok) * half + ip;
              csv[i] = e.rope_cos[o];
              snv[i] = e.rope_sin[o];
              slv[i] = k_tile ? e.slot_mapping[tok] : 0;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jj = c * 16 + i;
              xchg[i * kGemmTileN + f] = jj < m_valid ? v[i] * (scaled ? rs_s[jj] : 1.f) : 0.f;
            }
            named_barrier_sync(1, 128);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jj = c * 16 + i;
              if (jj >= m_valid) continue;
              const int tok = tok0 + jj;
              const float x = xchg[i * kGemmTileN + f], xp = xchg[i * kGemmTileN + partner];
              const float y = lo ? rope_lo(x, xp, csv[i], snv[i]) : rope_hi(xp, x, csv[i], snv[i]);
              if (!k_tile) {
                qo[static_cast<size_t>(tok) * e.q_dim + n0 + f] = Cvt<T>::from_f(y);
              } else {
                const long long slot = slv[i];
                if (slot < 0 || slot >= e.pool_slots) {
                  set_err(p.err, NS_DEV_BAD_SLOT);
                  continue;
                }
                const int col = n0 - e.q_dim + f;
                const size_t base = ((static_cast<size_t>(slot / e.block_size) * e.n_kv_heads + col / d) *
                                         e.block_size + static_cast<size_t>(slot % e.block_size)) * d;
                const T kv = Cvt<T>::from_f(y);
                kp[base + hf] = kv;
                if (e.kv_stage != nullptr)
                  reinterpret_cast<T*>(e.kv_stage)[static_cast<size_t>(tok) * 2 * e.kv_dim + col] = kv;
              }
            }
            named_barrier_sync(1, 128);
          } else if (p.epi == EPI_QKV) {
            // v columns
            T* vp = reinterpret_cast<T*>(e.v_pool);
            const int col = n0 - e.q_dim - e.kv_dim + f;
            const int kvh = col / d, dim = col - kvh * d;
            long long slv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) slv[i] = e.slot_mapping[tok0 + min(c * 16 + i, m_valid - 1)];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jj = c * 16 + i;
              if (jj >= m_valid) continue;
              const int tok = tok0 + jj;
              const long long slot = slv[i];
              if (slot < 0 || slot >= e.pool_slots) {
                set_err(p.err, NS_DEV_BAD_SLOT);
                continue;
              }
              const T val = Cvt<T>::from_f(v[i] * (scaled ? rs_s[jj] : 1.f));
              vp[((static_cast<size_t>(slot / e.block_size) * e.n_kv_heads + kvh) * e.block_size +
                  static_cast<size_t>(slot % e.block_size)) * d + dim] = val;
              if (e.kv_stage != nullptr)
                reinterpret_cast<T*>(e.kv_stage)[static_cast<size_t>(tok) * 2 * e.kv_dim + e.kv_dim + col] = val;
            }
          }
        }
        if (p.epi == EPI_RESID || p.epi == EPI_SWIGLU) fence_proxy_async_global();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[b]);
      }
      named_barrier_sync(1, 128);  // rs_s, xchg and the flag are reused by the next unit
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // Let this CTA's own copies in flight land before its shared memory is released.
    const int n_issued = *issued;
    for (int i = max(0, n_issued - ns); i < n_issued; ++i) {
      (void)mbar_wait(&full[i % ns], static_cast<uint32_t>(i / ns) & 1u, nullptr);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * ncols);
  }
}

// ------------------------------------------------------------------------------ host side

size_t gemm_smem_bytes(int BN, int nstage) {
  return 1024 + static_cast<size_t>(nstage) * (kABytes + static_cast<size_t>(BN) * kGemmTileK * 2) +
         kCtrlBytes;
}

namespace {

// Raise the kernels' dynamic shared-memory limit once per device (threads may race to do it;
// setting the attribute twice is harmless).
template <typename T>
cudaError_t gemm_configure() {
  static unsigned configured_mask = 0;  // accessed with atomic builtins
  int dev = 0;
  cudaGetDevice(&dev);
  const unsigned bit = dev < 31 ? 1u << dev : 0u;
  if (bit == 0 || !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_persistent_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured_mask, bit, __ATOMIC_RELEASE);
  }
  return cudaSuccess;
}

// How many clusters of `splits` CTAs with `smem` bytes of dynamic shared memory each the
// current device holds at once (the occupancy API places clusters within GPCs); cached.
int gemm_resident_clusters(int splits, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, splits, smem);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = 0;
  if (gemm_configure<__half>() == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, splits, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = splits;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<__half>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  std::lock_guard<std::mutex> g(mu);
  cache[key] = n;
  return n;
}

}  // namespace

int gemm_pick_stages(int BN, int kb_per_split, int clusters, int splits) {
  const size_t stage = kABytes + static_cast<size_t>(BN) * kGemmTileK * 2;
  // the epilogue tile [rows][128] fp32 reuses the stage ring
  const size_t tile_rows = gemm_two_pass(BN) ? kPassRows : BN;
  const int tile_min = static_cast<int>((tile_rows * kGemmTileN * 4 + stage - 1) / stage);
  const size_t half_sm = 113 * 1024 - 1024 - kCtrlBytes;
  // one CTA per SM: a deep ring keeps enough weight bytes in flight
  const size_t budget = 227 * 1024 - 1024 - kCtrlBytes;
  const int deep = std::max(std::min(static_cast<int>(budget / stage), 8),
                            std::max(tile_min, gemm_two_pass(BN) ? 2 : 4));
  // Half an SM: two CTAs per SM, one's epilogue overlapping the other's main loop; for decode
  // batches (narrow tiles) the next kernel's CTAs can be resident, streaming their own
  // weights, while this one runs.  As many stages as the CTA's k-range needs.
  const int half = std::max(std::min(static_cast<int>(half_sm / stage), std::max(kb_per_split, 2)),
                            std::max(tile_min, 2));
  if (BN <= 64) return half;
  // A wider tile takes the deep ring when the whole grid is resident with it in one wave (the
  // clusters placed as the hardware places them), else two per SM.
  return clusters <= gemm_resident_clusters(splits, gemm_smem_bytes(BN, deep)) ? deep : half;
}

uint32_t gemm_idesc(int dtype, int BN) {
  const uint32_t ab = dtype == NS_BF16 ? 1u : 0u;
  return (1u << 4)                                   // D format: fp32
         | (ab << 7) | (ab << 10)                    // A, B format: f16 / bf16
         | (static_cast<uint32_t>(BN >> 3) << 17)    // N >> 3
         | (static_cast<uint32_t>(kGemmTileN >> 4) << 24);  // M >> 4
}

namespace {
template <typename T>
cudaError_t launch_gemm_t(const CUtensorMap* mapA, const CUtensorMap* mapB, const GemmParams& p,
                          cudaStream_t s, bool pdl) {
  const size_t smem = gemm_smem_bytes(p.BN, p.nstage);
  cudaError_t e = gemm_configure<T>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.M + p.BN - 1) / p.BN, p.splits, p.N / kGemmTileN);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (p.splits > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = p.splits;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<T>, *mapA, *mapB, p);
}
}  // namespace

cudaError_t launch_gemm(const CUtensorMap* mapA, const CUtensorMap* mapB, const GemmParams& p,
                        int dtype, cudaStream_t s, bool pdl) {
  if (dtype == NS_BF16) return launch_gemm_t<__nv_bfloat16>(mapA, mapB, p, s, pdl);
  return launch_gemm_t<__half>(mapA, mapB, p, s, pdl);
}

namespace {
size_t gemm_persistent_smem(int BN, int nstage) {
  return 1024 + static_cast<size_t>(nstage) * (kABytes + static_cast<size_t>(BN) * kGemmTileK * 2) +
         kXchgFloats * sizeof(float) + kCtrlBytes;
}
}  // namespace

// As many stages as fit next to the exchange buffer and the control block (at most 8).
int gemm_persistent_stages(int BN) {
  const size_t stage = kABytes + static_cast<size_t>(BN) * kGemmTileK * 2;
  const size_t room = 227 * 1024 - 1024 - kXchgFloats * sizeof(float) - kCtrlBytes;
  return std::max(2, std::min(8, static_cast<int>(room / stage)));
}

namespace {
template <typename T>
cudaError_t launch_gemm_persistent_t(const CUtensorMap* mapA, const CUtensorMap* mapB, const GemmParams& p,
                                     int grid, cudaStream_t s, bool pdl) {
  cudaError_t e = gemm_configure<T>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = gemm_persistent_smem(p.BN, p.nstage);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<T>, *mapA, *mapB, p);
}
}  // namespace

cudaError_t launch_gemm_persistent(const CUtensorMap* mapA, const CUtensorMap* mapB, const GemmParams& p,
                                   int dtype, int grid, cudaStream_t s, bool pdl) {
  if (gemm_persistent_smem(p.BN, p.nstage) > 227 * 1024) return cudaErrorInvalidValue;
  if (dtype == NS_BF16) return launch_gemm_persistent_t<__nv_bfloat16>(mapA, mapB, p, grid, s, pdl);
  return launch_gemm_persistent_t<__half>(mapA, mapB, p, grid, s, pdl);
}

}  // namespace ns

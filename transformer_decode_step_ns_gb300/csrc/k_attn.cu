// Paged grouped-query decode attention: warp-independent units, cp.async-staged K/V tiles,
// tensor-core (mma.sync m16n8k16) QK^T and PV, split-K over fixed chunks with an in-kernel merge.
//
// "GPU waiting, not working" (nanoserve notes), change table: grouped-query attention must not
// materialise the G-times expanded copy of K and V, and one fused paged-attention kernel
// replaces about ten ops per layer.  "NanoFlow ..." ("Four resource classes"): decode attention
// is the memory-bound class, so the kernel is built to stream K/V at HBM speed:
//
// * Work unit = (request b, kv head g, superchunk).  A row's blocks split into superchunks of at
//   most 64 blocks (1024 tokens); the split is a function of the row's length alone, so a row's
//   result never depends on the rest of the batch.  A CTA takes a unit; its warps (8 at
//   head_dim 64, else 4) take contiguous shares of the superchunk and merge through shared
//   memory.
// * A CTA's first unit is its index.  When the launch holds at least kAttnQueueUnits units per
//   CTA, later units are handed out by a global counter as CTAs need them, rows with the
//   longest superchunks first (a stable counting sort that every CTA computes alike, so a unit
//   index names the same work everywhere): with a fixed round-robin deal the last CTA finished
//   12-16 % after the median one.  Below that the fixed deal over the rows in their own order
//   stays: CTA c takes units c, c + grid, c + 2 grid, ..., and since CTAs c and c + grid/2
//   share an SM, every SM gets the same number of units, while a queue can hand both CTAs of
//   one SM a second unit and leave another SM with none.  The two schedules are two compiled
//   variants (the queue's code slows the fixed deal's loop even unused); the host picks one.
//   Which CTA computes a unit does not change its result.  In the queue variant a superchunk of
//   fewer blocks than warps gives the extra warps a copy of a block to fetch and the empty
//   share's state to merge, so every warp streams every unit; the fixed deal skips such units.
// * Every warp streams its blocks (running ahead into its share of the CTA's next unit) through
//   a private ring of stages; each stage holds one 16 x d K tile and one V tile, copied with
//   16-byte cp.async by all 32 lanes (each tile is one contiguous run, so every warp request is a
//   coalesced 512-byte read) into an XOR-swizzled layout that keeps the ldmatrix reads below
//   bank-conflict free.  Small per-block copies go through the load/store path rather than the
//   TMA engine, whose per-request cost limits throughput at 2-4 KiB tiles.  The warp refills a
//   stage as soon as it has consumed it.
// * The G <= 8 query heads of the group form the rows of one 16-row mma.sync tile:
//     S^T[head][token]  = q[head][:] . K[token][:]          (A = q in registers, B = K tile)
//     O^T[dim][head]   += V^T[dim][token] . P^T[token][head] (A = V tile via ldmatrix.trans)
//   The accumulator layout of the first product is exactly the B-operand layout of the second,
//   so P never leaves registers.  Each K/V element is read once from shared memory for all G
//   heads: no expansion.  Online softmax in the log2 domain, per head, in registers.
// * The warps' shares are combined in warp order; superchunks of one (b, g) are combined by the
//   CTA that finishes last (atomic counter, no spin) in superchunk order with the log-sum-exp rule:
//   deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

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
  // warps per CTA; they split one superchunk (8 at head_dim 64, whose blocks are cheap to
  // stream but long to walk one by one)
  static constexpr int NW = D == 64 ? 8 : 4;
  static constexpr int NT = NW * 32;
  static constexpr int BS = 16;                // tokens per cache block
  static constexpr int NH = D / 64;            // 128-byte column halves of a tile
  static constexpr int TILE = BS * D * 2;      // bytes of one K or V tile
  static constexpr int STAGE = 2 * TILE;
  // stages per warp: G = 8 keeps the ring at two stages so two CTAs fit on an SM
  static constexpr int NST = (D == 128) ? (G == 8 ? 2 : 3) : 4;
  static constexpr int KS = D / 16;            // QK k-steps = PV m-tiles
  static constexpr int RING = NST * STAGE;     // bytes per warp
  static constexpr int CPL = 2 * BS * D / 8 / 32;  // 16-byte copies per lane per stage
  // CTA merge area: per warp acc [G][D] and (m, l) [G]; then merge weights [G][kAttnMaxChunks]
  static constexpr int OFF_MRG = NW * RING;
  static constexpr int MRG_FLOATS = NW * G * D + NW * G * 2 + 2 * G * kAttnMaxChunks + 4;  // + flag
  static constexpr int OFF_IDS = OFF_MRG + ((MRG_FLOATS * 4 + 15) & ~15);  // [NW][16] block ids
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(G >= 1 && G <= 8, "group");
  // then the CTA's unit sequence (SEQ 64-bit entries; the next index to claim and three spare
  // words); superchunk prefix over positions [batch + 1], row of each position [batch], the
  // warps' scan totals [NW], sort bins [NK].  The rows' lengths are read from seq_lens (it stays
  // in L1) rather than kept here: at head_dim 128 and a group of 4, two CTAs then share an SM up
  // to 665 rows.
  static constexpr int NK = kAttnSuperBlocks + 1;  // superchunk lengths 0 .. 64 (0: invalid row)
  static constexpr int SEQ = 16;
  static size_t smem_bytes(int batch) {
    return 1024 + OFF_IDS + NW * kAttnWarpBlocks * 4 +
           static_cast<size_t>(2 * batch + 1 + NW + NK + 2 * SEQ + 4) * 4;
  }
};

// Entry k of a CTA's unit sequence when it is not set yet (one lane; out of line, since it runs
// once per unit and the streaming loop around it is hot).  The first warp to get here claims the
// entry and takes the next ticket from the launch's counter; the others wait for it (bounded; a
// wait that runs out records NS_DEV_WAIT_TIMEOUT and ends the sequence).  Every CTA with a first
// unit takes exactly one ticket past the last unit, so the launch takes `total` tickets in all;
// the one that takes the last resets the counter (no CTA of this launch takes another, and the
// next launch reads it only after its dependency wait, when this grid has finished).
__device__ __noinline__ int queue_claim(unsigned long long* entry, int* claim, unsigned* sched,
                                        int total, int k, int* err) {
  volatile unsigned long long* e = entry;
  const unsigned long long tag = static_cast<unsigned long long>(k + 1) << 32;
  unsigned long long x;
  if (atomicCAS(claim, k, k + 1) == k) {
    const unsigned c = atomicAdd(sched, 1u);
    if (c == static_cast<unsigned>(total) - 1u) atomicExch(sched, 0u);
    x = tag | (gridDim.x + c);
    *e = x;
  } else {
    const unsigned long long t0 = global_timer_ns();
    while (((x = *e) >> 32) != static_cast<unsigned long long>(k + 1)) {
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        set_err(err, NS_DEV_WAIT_TIMEOUT);
        x = tag | 0x7fffffffu;
        break;
      }
    }
  }
  return static_cast<int>(x & 0x7fffffffu);
}

// Q: the launch may hand out units from the global queue (it does when it holds at least
// kAttnQueueUnits units per CTA).  Without Q the fixed deal is compiled alone: the queue's code
// in the same kernel slows the streaming loop even when it does not run.
template <typename T, int D, int G, bool Q>
__global__ void __launch_bounds__(AttnShape<D, G>::NT, AttnShape<D, G>::NW == 8 ? 1 : 2)
    attn_decode_kernel(const AttnParams p) {
  using S = AttnShape<D, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* m_acc = reinterpret_cast<float*>(smem + S::OFF_MRG);   // [NW][G][D]
  float* m_ml = m_acc + S::NW * G * D;                           // [NW][G][2]
  float* m_w = m_ml + S::NW * G * 2;                             // [2][G][kAttnMaxChunks]
  int* ids_all = reinterpret_cast<int*>(smem + S::OFF_IDS);      // [NW][kAttnWarpBlocks]
  // [SEQ] unit k of the CTA's sequence in entry k % SEQ, tagged (k + 1) << 32 | unit: one 64-bit
  // word, so a reader that sees the tag sees the unit without a fence
  unsigned long long* seq = reinterpret_cast<unsigned long long*>(ids_all + S::NW * kAttnWarpBlocks);
  int* seq_claim = reinterpret_cast<int*>(seq + S::SEQ);         // next sequence index to claim
  int* pre = seq_claim + 4;                                      // superchunk prefix [batch + 1]
  int* order = pre + p.batch + 1;                                // row of each position [batch]
  int* tot = order + p.batch;                                    // warp totals of the scan [NW]
  int* bins = tot + S::NW;                                       // [NK]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.n_kv_heads, batch = p.batch;
  uint8_t* ring = smem + warp * S::RING;
  if (Q && tid == 0) {
    for (int i = 1; i < S::SEQ; ++i) seq[i] = 0;
    // the first unit is fixed: it may be fetched before the dependency wait
    seq[0] = (1ull << 32) | blockIdx.x;
    *seq_claim = 1;
  }
  // Rows, their superchunk counts and the scheduling order.  seq_lens are step metadata, final
  // before the step starts, so under programmatic dependent launch this overlaps the previous
  // kernel.  Thread t validates rows [t * per, (t + 1) * per); a block-wide scan (warp shuffles,
  // then the warps' totals) counts the superchunks.  Without the queue the rows keep their order
  // and that scan is the prefix.  With it the rows are ordered longest superchunk first, ties by
  // row index (a stable counting sort): warp w ranks rows [w * wper, (w + 1) * wper), 32 at a
  // time; lanes holding the same length find each other with a match, and the warp's running
  // count per length (kept in the stage rings, free until the first copy) ranks them after its
  // earlier rows; order maps a position to its row.
  static_assert(S::NW * S::NK * 4 <= S::NW * S::RING && S::NK <= 96, "sort scratch");
  int* cnt = reinterpret_cast<int*>(smem);  // [NW][NK] a warp's rows per length (queue only)
  if (Q)
    for (int i = tid; i < S::NW * S::NK; i += S::NT) cnt[i] = 0;
  auto row_len = [&](int b) {  // the row's length, 0 when outside [1, mb * block_size]
    const int L = __ldg(p.seq_lens + p.row0 + b);
    return L >= 1 && L <= p.mb * p.block_size ? L : 0;
  };
  auto block_scan = [&](int v) {  // inclusive over the warp; lane 31 leaves the warp's total
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) tot[warp] = inc;
    return inc;
  };
  const int per = (batch + S::NT - 1) / S::NT;
  const int lo_t = tid * per, hi_t = min(batch, lo_t + per);
  int run = 0;
  for (int b = lo_t; b < hi_t; ++b) {
    const int L0 = row_len(b);
    if (L0 == 0) set_err(p.err, NS_DEV_BAD_LENGTH);
    run += L0 > 0 ? attn_num_chunks(L0) : 0;
  }
  int inc = block_scan(run);
  __syncthreads();
  int before_warp = 0, n_chunks = 0;
  for (int w = 0; w < S::NW; ++w) {
    const int t = tot[w];
    before_warp += w < warp ? t : 0;
    n_chunks += t;
  }
  const bool queue = Q && static_cast<long long>(n_chunks) * Hkv >=
                              static_cast<long long>(kAttnQueueUnits) * gridDim.x;  // block-uniform
  if (queue) {
    const int wper = (batch + S::NW - 1) / S::NW;
    const int lo = warp * wper, hi = min(batch, lo + wper);
    int* wc = cnt + warp * S::NK;
    for (int b0 = lo; b0 < hi; b0 += 32) {
      const int b = b0 + lane;
      const unsigned act = __ballot_sync(0xffffffffu, b < hi);
      if (b < hi) {
        const int key = attn_chunk_blocks(row_len(b));
        const unsigned same = __match_any_sync(act, key);
        const int before = __popc(same & ((1u << lane) - 1u));
        pre[b] = wc[key] + before;  // rank among this warp's rows of the same length
        __syncwarp(act);
        if (before == 0) wc[key] += __popc(same);
      }
      __syncwarp();
    }
    __syncthreads();
    if (tid < S::NK) {  // per length: the warps' offsets, and the length's total
      int acc = 0;
      for (int w = 0; w < S::NW; ++w) {
        const int v = cnt[w * S::NK + tid];
        cnt[w * S::NK + tid] = acc;
        acc += v;
      }
      bins[tid] = acc;
    }
    __syncthreads();
    if (warp == 0) {  // where each length starts, longest first (lane l: the 3l-th to 3l+2-th)
      int v[3], sum = 0;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int k = S::NK - 1 - (3 * lane + j);
        v[j] = k >= 0 ? bins[k] : 0;
        sum += v[j];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int acc = incl - sum;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int k = S::NK - 1 - (3 * lane + j);
        if (k >= 0) bins[k] = acc;
        acc += v[j];
      }
    }
    __syncthreads();
    for (int b0 = lo; b0 < hi; b0 += 32) {
      const int b = b0 + lane;
      if (b < hi) {
        const int key = attn_chunk_blocks(row_len(b));
        order[bins[key] + wc[key] + pre[b]] = b;
      }
    }
    __syncthreads();
    // the superchunk counts again, now over positions
    run = 0;
    for (int i = lo_t; i < hi_t; ++i) run += attn_num_chunks(row_len(order[i]));
    inc = block_scan(run);
    __syncthreads();
    before_warp = 0;
    for (int w = 0; w < warp; ++w) before_warp += tot[w];
  }
  {
    int acc = before_warp + inc - run;
    for (int i = lo_t; i < hi_t; ++i) {
      pre[i] = acc;
      acc += attn_num_chunks(row_len(queue ? order[i] : i));
    }
    if (tid == S::NT - 1) pre[batch] = acc;
    __syncthreads();
  }
  const int total = pre[batch] * Hkv;
  if (tid == 0) griddep_launch_dependents();

  // A unit is (row b, kv head g, superchunk sc); this warp's share is blocks [w0, w1) of it.
  struct Unit {
    int b, g, sc, L, blk0, nchunks, w0, w1;
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
    x.b = queue ? order[lo] : lo;
    x.sc = cg - pre[lo];
    x.L = row_len(x.b);
    x.nchunks = attn_num_chunks(x.L);
    const int cb = attn_chunk_blocks(x.L);
    x.blk0 = x.sc * cb;
    const int nb = min(cb, (x.L + S::BS - 1) / S::BS - x.blk0);
    x.w0 = x.blk0 + (nb * warp) / S::NW;
    x.w1 = x.blk0 + (nb * (warp + 1)) / S::NW;
    // With the queue a warp whose share would be empty (fewer blocks than warps) fetches one
    // block of another warp's share and merges the empty share's state instead, so every warp
    // streams every unit.  The fixed deal skips such units.
    if constexpr (Q) x.w1 = max(x.w1, x.w0 + 1);
    return x;
  };

  // ---- producer cursor (warp-uniform): this warp's stream of blocks over its units, in
  // consumption order.  The block ids of the next unit are loaded into a register when the
  // producer enters the current one and stored to shared memory when it gets there, so the
  // stream never waits on a block-table read.  Every stage is one cp.async group, so "oldest
  // stage landed" is wait_group(NST - 1).
  int* ids = ids_all + warp * kAttnWarpBlocks;
  const uint64_t pol = policy_evict_first();  // K/V are streamed once
  const T* kpool = reinterpret_cast<const T*>(p.k_pool);
  const T* vpool = reinterpret_cast<const T*>(p.v_pool);
  // Unit k of this CTA's sequence (warp-collective).  The first warp that needs an entry not yet
  // set claims it and takes the next unit from the global counter; the others wait for it
  // (bounded).  Every warp has blocks in every unit and the warps merge each unit before the
  // next, so a producer leads the slowest consumer by at most NST + 1 units and an entry is not
  // reused (SEQ units later) while any warp still needs it.
  auto unit_at = [&](int k) -> int {
    if (!queue) return blockIdx.x + k * gridDim.x;
    int v = 0;
    if (lane == 0) {
      const unsigned long long x = *(volatile unsigned long long*)(seq + k % S::SEQ);
      v = (x >> 32) == static_cast<unsigned long long>(k + 1)
              ? static_cast<int>(x & 0x7fffffffu)
              : queue_claim(seq + k % S::SEQ, seq_claim, p.sched, total, k, p.err);
    }
    return __shfl_sync(0xffffffffu, v, 0);
  };
  int pk = 0, pu = blockIdx.x, pi = 0, nxt = 0x7fffffff;
  bool lookahead = !queue;  // later units may be named (with the queue: after the dependency wait)
  Unit pun{}, nun{};
  int nid = 0;
  auto load_ids = [&](int unit) {  // register <- this warp's block ids of `unit` (non-blocking)
    nun = decode(unit);
    const int* src = p.block_tables + static_cast<size_t>(p.row0 + nun.b) * p.mb;
    nid = lane < nun.w1 - nun.w0 ? src[nun.w0 + lane] : 0;
  };
  auto enter = [&]() {  // the producer moves to unit pu (decoded in nun)
    for (;;) {
      __syncwarp();
      if (pu >= total) break;
      pun = nun;
      if (lane < pun.w1 - pun.w0) {
        int blk = nid;
        if (blk < 0 || blk >= p.num_blocks) {
          set_err(p.err, NS_DEV_BAD_BLOCK);
          blk = 0;  // keep the pipeline consistent; the error word flags the result
        }
        ids[lane] = blk;
      }
      if constexpr (Q) {  // every share is non-empty
        if (lookahead) {
          nxt = unit_at(pk + 1);
          if (nxt < total) load_ids(nxt);
        }
        __syncwarp();
        break;
      } else {  // units where this warp has no blocks are skipped
        if (pu + static_cast<int>(gridDim.x) < total) load_ids(pu + gridDim.x);
        __syncwarp();
        if (pun.w1 > pun.w0) break;
        pu += gridDim.x;
      }
    }
  };
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
      if (++pi >= pun.w1 - pun.w0) {
        pi = 0;
        if constexpr (Q) {
          pk += 1;
          pu = nxt;
        } else {
          pu += gridDim.x;
        }
        enter();
      }
    }
    cp_async_commit();
  };
  if (pu < total) load_ids(pu);
  enter();
  // Blocks without a token of this step may be fetched before the previous kernel (which writes
  // this step's K/V and q) has finished.  In a decode-only batch only the last block of a row
  // holds this step's token; rows of a prefill chunk read blocks other rows write now, and the
  // host then clears early_ok.  With the queue the early fetches stay inside the first unit:
  // the counter that hands out later units may still be in use by the previous launch until the
  // dependency wait.
  const bool early = p.early_ok == nullptr || *p.early_ok != 0;
  int s0 = 0;
  while (early && s0 < S::NST && pu < total && pun.w0 + pi != (pun.L - 1) / S::BS &&
         (!queue || pi + 1 < pun.w1 - pun.w0))
    issue(s0++);
  griddep_wait();
  lookahead = true;
  if (queue && pu < total) {  // the early fetches stayed in the first unit
    nxt = unit_at(1);
    if (nxt < total) load_ids(nxt);
  }
  for (int s = s0; s < S::NST; ++s) issue(s);

  const int gq = lane >> 2, tq = lane & 3;
  // ldmatrix lane address: token row and 16-byte chunk offset within the 4 matrices
  const int lm_tok = (lane & 7) + ((lane >> 4) << 3);
  const int lm_chunk = (lane >> 3) & 1;
  T* out = reinterpret_cast<T*>(p.out);
  const int h_e = 2 * tq, h_o = 2 * tq + 1;

  int ci = 0;
  for (int k = 0;; ++k) {
    const int u = unit_at(k);
    if (u >= total) break;
    const Unit x = decode(u);
    const size_t row = static_cast<size_t>(p.row0 + x.b);
    float m_run = -INFINITY, l_run = 0.f;
    float acc[S::KS][4];
#pragma unroll
    for (int mt = 0; mt < S::KS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    if (Q || x.w1 > x.w0) {
      // q of the group as the A operand: rows = heads (G of 16 used), k = dims
      uint32_t qa[S::KS][2];
      {
        const T* qrow = reinterpret_cast<const T*>(p.q) + row * p.q_row_stride +
                        static_cast<size_t>(x.g * G + (gq < G ? gq : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < S::KS; ++ks) {
          qa[ks][0] = gq < G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tq) : 0u;
          qa[ks][1] = gq < G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tq) : 0u;
        }
      }
      for (int i = x.w0; i < x.w1; ++i, ++ci) {
        const int s = ci % S::NST;
        cp_async_wait_group<S::NST - 1>();  // this lane's copies of the oldest stage landed
        __syncwarp();                       // ... and every other lane's
        const uint8_t* kt = ring + s * S::STAGE;
        const uint8_t* vt = kt + S::TILE;
        const int n_valid = min(S::BS, x.L - i * S::BS);
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
    }

    // ---- merge the warps' shares of the superchunk through shared memory, in warp order
    {
      // a warp that streamed a copy (its own share was empty) gives the empty share's state
      const int nb = min(attn_chunk_blocks(x.L), (x.L + S::BS - 1) / S::BS - x.blk0);
      if (Q && (nb * (warp + 1)) / S::NW == (nb * warp) / S::NW) {
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int mt = 0; mt < S::KS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      }
      float* wacc = m_acc + warp * G * D;
#pragma unroll
      for (int mt = 0; mt < S::KS; ++mt) {
        const int d0 = mt * 16 + gq;
        if (h_e < G) {
          wacc[h_e * D + d0] = acc[mt][0];
          wacc[h_e * D + d0 + 8] = acc[mt][2];
        }
        if (h_o < G) {
          wacc[h_o * D + d0] = acc[mt][1];
          wacc[h_o * D + d0 + 8] = acc[mt][3];
        }
      }
      if (tq == 0 && gq < G) {
        m_ml[(warp * G + gq) * 2] = m_run;
        m_ml[(warp * G + gq) * 2 + 1] = l_run;
      }
    }
    named_barrier_sync(1, S::NT);
    // combined (m, l) of the superchunk per head, and each warp's weight 2^(m_w - M)
    float* pacc = p.partials + (row * Hkv + x.g) * attn_slot_floats(p.max_chunks, G, D);
    float* pml = pacc + static_cast<size_t>(p.max_chunks) * G * D;
    for (int e = tid; e < G * D; e += S::NT) {
      const int hh = e / D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < S::NW; ++w) M = fmaxf(M, m_ml[(w * G + hh) * 2]);
      float o = 0.f, Ls = 0.f;
#pragma unroll
      for (int w = 0; w < S::NW; ++w) {
        const float wt = M == -INFINITY ? 0.f : exp2f(m_ml[(w * G + hh) * 2] - M);
        o = fmaf(m_acc[(w * G) * D + e], wt, o);
        Ls = fmaf(m_ml[(w * G + hh) * 2 + 1], wt, Ls);
      }
      if (x.nchunks == 1) {
        out[row * p.out_row_stride + static_cast<size_t>(x.g) * G * D + e] = MV<T>::from_f(o / Ls);
      } else {
        pacc[static_cast<size_t>(x.sc) * G * D + e] = o;
        if ((e % D) == 0) reinterpret_cast<float2*>(pml)[x.sc * G + hh] = make_float2(M, Ls);
      }
    }
    if (x.nchunks > 1) {
      // Superchunks of one (row, kv head) are merged by the CTA that finishes last.  The barrier
      // orders every thread's partial stores before thread 0's increment, which releases them
      // at GPU scope and acquires the other CTAs' (acq_rel); the second barrier passes that on
      // to the threads that read them.  No thread fences while its copies are in flight.
      named_barrier_sync(1, S::NT);
      int* last_flag = reinterpret_cast<int*>(m_w + 2 * G * kAttnMaxChunks);
      if (tid == 0) {
        int* cnt = p.counters + row * Hkv + x.g;
        int prev;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(prev) : "l"(cnt) : "memory");
        const int last = prev == x.nchunks - 1 ? 1 : 0;
        if (last) *cnt = 0;  // ready for the next launch
        last_flag[0] = last;
      }
      named_barrier_sync(1, S::NT);
      if (last_flag[0]) {
        // weight_c = 2^(m_c - M) / sum_c' l_c' 2^(m_c' - M), summed in superchunk order
        float* wm = m_w;                          // [G][kAttnMaxChunks]: m, then the weight
        float* wl = m_w + G * kAttnMaxChunks;     // [G][kAttnMaxChunks]: l
        for (int i = tid; i < x.nchunks * G; i += S::NT) {
          const float2 v = __ldcg(reinterpret_cast<const float2*>(pml) + i);
          const int c = i / G, hh = i - c * G;
          wm[hh * kAttnMaxChunks + c] = v.x;
          wl[hh * kAttnMaxChunks + c] = v.y;
        }
        named_barrier_sync(1, S::NT);
        if (tid < G) {
          float M = -INFINITY;
          for (int c = 0; c < x.nchunks; ++c) M = fmaxf(M, wm[tid * kAttnMaxChunks + c]);
          float Ls = 0.f;
          for (int c = 0; c < x.nchunks; ++c)
            Ls = fmaf(wl[tid * kAttnMaxChunks + c], exp2f(wm[tid * kAttnMaxChunks + c] - M), Ls);
          const float inv = 1.f / Ls;
          for (int c = 0; c < x.nchunks; ++c)
            wm[tid * kAttnMaxChunks + c] = exp2f(wm[tid * kAttnMaxChunks + c] - M) * inv;
        }
        named_barrier_sync(1, S::NT);
        T* orow = out + row * p.out_row_stride + static_cast<size_t>(x.g) * G * D;
        constexpr int NC4 = G * D / 4;
        for (int col = tid; col < NC4; col += S::NT) {
          const int hh = col / (D / 4), dq = col - hh * (D / 4);
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int cb = 0; cb < x.nchunks; cb += 8) {  // 8 superchunks' loads in flight at a time
            float4 v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
              if (cb + c < x.nchunks)
                v[c] = __ldcg(reinterpret_cast<const float4*>(pacc + (static_cast<size_t>(cb + c) * G + hh) * D) + dq);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              if (cb + c < x.nchunks) {
                const float w = wm[hh * kAttnMaxChunks + cb + c];
                o.x = fmaf(v[c].x, w, o.x);
                o.y = fmaf(v[c].y, w, o.y);
                o.z = fmaf(v[c].z, w, o.z);
                o.w = fmaf(v[c].w, w, o.w);
              }
            }
          }
          T* dst = orow + hh * D + 4 * dq;
          dst[0] = MV<T>::from_f(o.x);
          dst[1] = MV<T>::from_f(o.y);
          dst[2] = MV<T>::from_f(o.z);
          dst[3] = MV<T>::from_f(o.w);
        }
      }
    }
    named_barrier_sync(1, S::NT);  // the merge area is reused by the next unit
  }
  cp_async_wait_group<0>();  // every copy this warp issued was consumed; drain regardless
}

// ------------------------------------------------------------------------------ host side

}  // namespace ns

#include <map>
#include <mutex>
#include <utility>

namespace ns {

namespace {

template <typename T, int D, int G, bool Q>
cudaError_t launch_attn_t(const AttnParams& p, int grid, cudaStream_t s, bool pdl) {
  using S = AttnShape<D, G>;
  static int configured_mask = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 31 && !(configured_mask & (1 << dev))) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<T, D, G, Q>,
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
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<T, D, G, Q>, p);
}

template <typename T, int D, bool Q>
cudaError_t dispatch_g(const AttnParams& p, int group, int grid, cudaStream_t s, bool pdl) {
  switch (group) {
    case 1: return launch_attn_t<T, D, 1, Q>(p, grid, s, pdl);
    case 2: return launch_attn_t<T, D, 2, Q>(p, grid, s, pdl);
    case 4: return launch_attn_t<T, D, 4, Q>(p, grid, s, pdl);
    case 7: return launch_attn_t<T, D, 7, Q>(p, grid, s, pdl);
    case 8: return launch_attn_t<T, D, 8, Q>(p, grid, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D>
cudaError_t dispatch_q(const AttnParams& p, int group, int grid, cudaStream_t s, bool pdl,
                       bool queue) {
  return queue ? dispatch_g<T, D, true>(p, group, grid, s, pdl)
               : dispatch_g<T, D, false>(p, group, grid, s, pdl);
}

// One full wave of the kernel for `batch` rows on the current device: SMs x resident CTAs per
// SM, asked of the occupancy API once per (device, shared memory size) and kept.
template <typename T, int D, int G>
int max_grid_t(int batch) {
  using S = AttnShape<D, G>;
  static std::mutex mu;
  static std::map<std::pair<int, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_pair(dev, S::smem_bytes(batch));
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int sms = 1, per_sm = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // both variants: the same block size, shared memory and register bound
  int per_sm_q = 0;
  cudaFuncSetAttribute(attn_decode_kernel<T, D, G, false>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  cudaFuncSetAttribute(attn_decode_kernel<T, D, G, true>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_decode_kernel<T, D, G, false>,
                                                    S::NT, S::smem_bytes(batch)) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_q, attn_decode_kernel<T, D, G, true>,
                                                    S::NT, S::smem_bytes(batch)) != cudaSuccess)
    per_sm = per_sm_q = 1;
  per_sm = std::max(1, std::min(per_sm, per_sm_q));
  std::lock_guard<std::mutex> g(mu);
  cache[key] = sms * per_sm;
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
                        cudaStream_t s, bool pdl, bool queue) {
  if (grid < 1) grid = 1;
  if (dtype == NS_BF16) {
    return head_dim == 64 ? dispatch_q<__nv_bfloat16, 64>(p, group, grid, s, pdl, queue)
                          : dispatch_q<__nv_bfloat16, 128>(p, group, grid, s, pdl, queue);
  }
  return head_dim == 64 ? dispatch_q<__half, 64>(p, group, grid, s, pdl, queue)
                        : dispatch_q<__half, 128>(p, group, grid, s, pdl, queue);
}

}  // namespace ns

// Types and inline functions shared by the kernels and the host runtime (ns_api.cu): parameter
// blocks, tile constants and the attention split.  Host-only declarations are in ns_host.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ns.h"

namespace ns {

constexpr int kGemmTileN = 128;   // output features per CTA (UMMA M)
constexpr int kGemmTileK = 64;    // K per pipeline stage (one 128-byte swizzle row)
constexpr int kGemmThreads = 192; // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kMaxBN = 256;       // token tile (UMMA N) upper bound
constexpr int kMaxSplits = 8;     // split-K CTAs per tile = portable cluster size
constexpr int kAttnSuperBlocks = 64;  // decode attention: rows split into superchunks of <= 64 blocks
constexpr int kAttnMaxChunks = 64;    // superchunks per row (seq_len <= 65536 with 16-token blocks)
constexpr int kAttnWarpBlocks = 16;   // block ids one warp holds per superchunk (64 / 4 warps at
                                      // most; 8 at head_dim 64)
// Decode attention units (row, kv head, superchunk) per CTA from which a launch hands out its
// later units from a global queue, longest superchunks first, instead of a fixed deal (measured
// on the paged attention benchmark: at 4-6 units per CTA the two tie, at 1-3 the fixed deal is
// 8-14 % faster, from 10 the queue is 4-7 % faster).
constexpr int kAttnQueueUnits = 6;
constexpr int kMaxRows = 4096;

enum EpiMode : int {
  EPI_F32 = 0,     // y = acc (* rs) -> fp32 [tok][ldo]
  EPI_QKV = 1,     // rs scale, RoPE on q/k, q -> q_out, k/v -> paged pools at slot_mapping
  EPI_RESID = 2,   // resid += acc; xn = resid * gamma_next; per-tile sum of squares
  EPI_SWIGLU = 3,  // rows [0,64) gate, [64,128) up: act = silu(rs g) * (rs u)
};

struct EpiArgs {
  // fused RMSNorm scale: rs[tok] = rsqrt(sum_t sumsq_in[t * sumsq_ld + tok] / norm_dim + eps)
  const float* sumsq_in;
  int sumsq_tiles, sumsq_ld, norm_dim;
  float eps;
  // EPI_F32
  float* out_f32;
  long long ldo;
  const unsigned long long* out_ptr_slot;  // when set, the output base is read from here
  const int* rows_valid;                   // when set, rows at or past *rows_valid are padding
  // EPI_QKV
  void* q_out;
  void* k_pool;
  void* v_pool;
  const long long* slot_mapping;
  const float* rope_cos;
  const float* rope_sin;
  int q_dim, kv_dim, head_dim, n_kv_heads, block_size;
  long long pool_slots;
  void* kv_stage;  // when set, row `tok` of [rows][2][kv_dim] also receives the K and V it writes
  // EPI_RESID
  float* resid;
  void* xn_out;
  const float* gamma_next;
  float* sumsq_out;
  int resid_dim;
  // EPI_SWIGLU
  void* act_out;
  int ffn;
};

struct GemmParams {
  int M;        // rows (tokens) in this launch
  int row0;     // first row in the activation / output buffers
  int N, K;     // output features, reduction length
  int BN;       // token tile, multiple of 16, 16..256
  int splits;   // split-K count = cluster size along grid y (<= kMaxSplits)
  int kb_per_split;
  int nstage;
  int epi;
  uint32_t idesc;
  int* err;
  EpiArgs e;
  int tiles_m;  // persistent variant: token tiles of BN rows
};

// Launches of fewer rows than this take the persistent GEMM only when they are very long.
constexpr int kPersistentMinRows = 65;

struct AttnParams {
  const void* q;
  long long q_row_stride;  // elements between rows of q
  const void* k_pool;
  const void* v_pool;
  const int* block_tables;
  int mb;                  // block-table row width
  const int* seq_lens;
  void* out;
  long long out_row_stride;
  int batch, row0, n_kv_heads, num_blocks, block_size;
  float scale_log2;        // softmax scale * log2(e)
  int max_chunks;          // partial slots per (row, kv head): attn_max_chunks(mb * block_size)
  float* partials;         // per (row, kv head), attn_slot_floats apart (16-byte aligned):
                           // [max_chunks][G][head_dim] accumulators, then [max_chunks][G][2] (m, l)
  int* counters;           // [rows][n_kv_heads], zero between launches
  // the attention unit queue's ticket counter: zero at launch, and zero again when the launch
  // has taken its last ticket.  Launches that may run at the same time use different words.
  unsigned* sched;
  int* err;
  // Device word, read before the dependency wait: nonzero when no block a row reads, other than
  // its last, receives a token in this step, so those blocks may be fetched while the previous
  // kernel (which writes this step's K/V) still runs.  nullptr = always (K/V are inputs).
  const int* early_ok;
};

// Causal attention of a prefill chunk: rows row0 .. row0 + chunk - 1 of the batch are queries at
// consecutive positions (positions[row0] first) over the block table of row table_row.
struct PrefillParams {
  const void* q;
  long long q_row_stride;
  const void* k_pool;
  const void* v_pool;
  const int* block_tables;
  int mb;
  int table_row;        // the chunk row whose table covers every position of the chunk
  const int* positions;
  void* out;
  long long out_row_stride;
  int row0, chunk, n_kv_heads, num_blocks;
  float scale_log2;
  int* err;
};

// A run of at least this many rows at consecutive positions over one block table at the end of
// a step is attended as a prefill chunk.
constexpr int kPrefillMinRows = 16;

struct EmbedParams {
  const void* embed;
  const int* token_ids;   // step metadata; an id -(r + 1) names row r of tok_src
  const int* tok_src;     // device token source (ns_set_token_source) or null
  const int* positions;
  int vocab, hidden;
  const float* gamma;  // first layer's attention-norm gain (fp32)
  float* resid;
  void* xn;
  float* sumsq;
  int sumsq_ld;
  float* rope_cos;
  float* rope_sin;
  int head_dim;
  const double* inv_freq;  // [head_dim / 2] theta^(-2i/d), fp64
  int batch, row0;
  const int* rows_valid;  // when set, rows at or past *rows_valid are padding (token 0)
  int* err;
};

// A GEMM tile wider than kPassRows tokens stages its accumulator in shared memory
// kPassRows tokens at a time, so its stage ring may be two stages (two CTAs per SM).
constexpr int kPassRows = 128;
__host__ __device__ inline bool gemm_two_pass(int BN) { return BN > kPassRows; }

// Split of a row of length L (a function of L alone, 16-token blocks): ceil(L / 16) blocks in
// ceil(blocks / 64) superchunks of ceil(blocks / superchunks) blocks; a CTA's warps share one
// superchunk.  attn_max_chunks bounds the superchunk count of any L <= L_max.
__host__ __device__ inline int attn_num_chunks(int L) {
  return L <= 0 ? 0 : ((L + 15) / 16 + kAttnSuperBlocks - 1) / kAttnSuperBlocks;
}
__host__ __device__ inline int attn_chunk_blocks(int L) {
  const int nb = (L + 15) / 16, n = attn_num_chunks(L);
  return n == 0 ? 0 : (nb + n - 1) / n;
}
// Floats of one (row, kv head) partial slot, rounded up so every slot starts 16-byte aligned.
__host__ __device__ inline size_t attn_slot_floats(int max_chunks, int group, int head_dim) {
  return (static_cast<size_t>(max_chunks) * group * (head_dim + 2) + 3) & ~static_cast<size_t>(3);
}
__host__ __device__ inline int attn_max_chunks(int L_max) {
  const int c = attn_num_chunks(L_max);
  return c < 1 ? 1 : (c < kAttnMaxChunks ? c : kAttnMaxChunks);
}

// ------------------------------------------------------------------ persistent step kernel
// One cooperative launch runs a whole decode step of at most kStepMaxRows rows (k_step.cu).
constexpr int kStepMaxRows = 32;
// 7 compute warps + 1 weight-streaming warp: with 8 warps each of the SM's four register-file
// partitions holds two warps, so a thread may use up to 255 registers.
constexpr int kStepWarps = 7;                          // compute warps
constexpr int kStepThreads = (kStepWarps + 1) * 32;    // + one weight-streaming warp
constexpr int kStepChunk = 4096;                       // bytes of one weight chunk: 16 x 128
// Ring slots hold kStepSlotChunks consecutive chunks, fetched by one bulk copy: measured on
// GB300, 4 KiB TMA bulk copies stream at most ~16 GB/s per SM (their per-request cost), 16 KiB
// copies ~47 GB/s per SM (the HBM share of an SM).
constexpr int kStepSlotChunks = 4;
constexpr int kStepSlot = kStepChunk * kStepSlotChunks;
constexpr int kStepGroup = 2;                          // output tiles reduced together
constexpr int kStepAttnBlocks = 2 * kStepWarps;        // cache blocks per attention unit
constexpr int kStepRedStride = 24;                     // floats per token row of a reduced tile
// A stage copies the activation columns it reduces over, for every row, into shared memory with
// one bulk copy; at most kStepSliceChunks 128-column chunks (64 KiB at 32 rows).  Longer
// reductions are split over teams of CTAs (split-K), the splits summed in split order.
constexpr int kStepSliceChunks = 8;
constexpr int kStepActBytes = kStepSliceChunks * kStepMaxRows * 256;
constexpr int kStepMaxTilesPerCta = 32;                // tiles of one split stage per CTA

enum StepStage : int { SS_QKV = 0, SS_O = 1, SS_GU = 2, SS_DOWN = 3, SS_LM = 4, SS_COUNT = 5 };

// How one 16-row output tile of a projection maps to weight rows.
enum PackKind : int {
  PK_PLAIN = 0,  // rows row0 .. row0 + 15
  PK_ROPE = 1,   // q/k head tile: rows 0-7 are features j*8.. of the head's first half, rows
                 // 8-15 the same features of its second half (RoPE partners)
  PK_GU = 2,     // rows 0-7 gate features j*8.., rows 8-15 the same up features
};

// One 4 KiB chunk of the packed weight stream: tile `tile` of matrix `w` (K columns),
// columns kc*128 .. kc*128 + 127.
struct PackDesc {
  const void* w;
  int K, kind, tile, kc, row0, pad;
};

// The output tiles one CTA computes in a stage: tiles first, first + stride, ... (count of them)
// over columns [kc0, kc1) of the reduction (split `split` of the stage).  An unsplit stage deals
// its tiles round-robin from CTA `rot`; a stage split S ways forms teams of S consecutive CTAs,
// team q taking tiles q, q + teams, ... and member s the s-th column range.
struct StepTiles {
  int first, stride, count, split, kc0, kc1;
};
__host__ __device__ inline StepTiles step_tiles(int grid, int cta, int n_tiles, int kc, int S, int rot) {
  StepTiles t{0, 1, 0, 0, 0, kc};
  if (S <= 1) {
    t.first = (cta - rot % grid + grid) % grid;
    t.stride = grid;
    t.count = t.first < n_tiles ? (n_tiles - t.first + grid - 1) / grid : 0;
    return t;
  }
  const int teams = grid / S;
  if (cta >= teams * S) return t;
  const int q = cta / S;
  t.split = cta - q * S;
  t.first = q;
  t.stride = teams;
  t.count = q < n_tiles ? (n_tiles - q + teams - 1) / teams : 0;
  t.kc0 = t.split * kc / S;
  t.kc1 = (t.split + 1) * kc / S;
  return t;
}

struct StepParams {
  int B;  // rows of the step (<= kStepMaxRows)
  int H, qd, kvd, F, vocab, d, G, Hq, Hkv, n_layers;
  float eps, scale_log2;
  int nslot;    // weight ring slots of kStepSlot bytes
  int with_lm;  // 0: the step ends after the last layer
  // per stage: output tiles, 128-column chunks of the reduction, K splits, round-robin start
  int n_tiles[SS_COUNT], kc[SS_COUNT], split[SS_COUNT], rot[SS_COUNT];
  int max_split_tiles;  // counter slots per (layer, stage) of the split stages
  // packed weights: CTA c streams chunks stream_off[c] .. stream_off[c + 1] - 1 of wpack, its
  // LM-head chunks from stream_lm[c]
  const uint8_t* wpack;
  const long long* stream_off;
  const long long* stream_lm;
  const void* embed;
  const float* attn_norm;   // [n_layers][H]
  const float* ffn_norm;    // [n_layers][H]
  const float* final_norm;  // [H]
  uint8_t* pools;           // K of layer l at 2l * pool_bytes, V at (2l + 1) * pool_bytes
  size_t pool_bytes;
  int num_blocks, mb, block_size;
  long long pool_slots;
  // step metadata
  const int* tok;
  const int* tok_src;
  const int* pos;
  const int* seq;
  const long long* slot;
  const int* tab;
  const unsigned long long* logits_slot;
  const int* rows_valid;
  const int* early_ok;  // see AttnParams::early_ok
  const double* inv_freq;
  // activations: resid fp32 [rows][H]; xn, o, act chunk-major [width / 128][B][128] (every
  // column slice of all rows is contiguous); q row-major [rows][qd]; per-16-column sums of
  // squares of the residual [rows][H / 16]
  float* resid;
  void* xn;
  void* q;
  void* o;
  void* act;
  float* sumsq16;
  // split-K partial tiles [tile][split][kStepMaxRows][16] fp32
  float* split_part;
  // attention partials [kStepMaxRows][Hkv][max_ch][G][d + 2]
  float* attn_part;
  int max_ch;
  // [0] barrier arrivals, [1] abort flag, [2..] attention unit counters
  // [n_layers][kStepMaxRows][Hkv], then split-K tile counters [n_layers + 1][4][max_split_tiles];
  // zero at launch
  unsigned* sync;
  int* err;
};

// Copy between the paged pools and a contiguous buffer [n_layers][n][2][kv_dim] whose row
// (layer, t) holds the K then V of the token at slot slots[t] (see ns_kv_reload / ns_kv_save).
struct KvCopyParams {
  void* pools;              // 2 * n_layers pools of pool_bytes: K of layer l at 2l, V at 2l + 1
  size_t pool_bytes;
  void* buf;                // contiguous rows, 16-byte aligned
  const long long* slots;   // [n], device
  int n, n_layers, n_kv_heads, head_dim, block_size;
  long long pool_slots;     // slots at or past this are refused (error flag, no access)
  int to_pool;              // 1: buf -> pages, 0: pages -> buf
  int* err;
};

}  // namespace ns

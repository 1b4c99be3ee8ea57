// Host-side interfaces of the kernel files, used by the runtime (ns_api.cu, ns_noalloc.cu,
// ns_sched.cpp): launchers, launch-shape choices and the error-message setter.  Device code
// does not depend on this file.
#pragma once

#include <vector>

#include "ns_internal.h"

namespace ns {

// Kernel launchers return the launch error; `pdl` adds programmatic stream serialisation.
size_t gemm_smem_bytes(int BN, int nstage);
// Stage-ring depth for a launch of `clusters` clusters of `splits` CTAs (the depth never changes
// results).
int gemm_pick_stages(int BN, int kb_per_split, int clusters, int splits);
uint32_t gemm_idesc(int dtype, int BN);
cudaError_t launch_gemm(const CUtensorMap* mapA, const CUtensorMap* mapB, const GemmParams& p,
                        int dtype, cudaStream_t s, bool pdl);
// Persistent variant for unsplit weights: `grid` CTAs (at most one per SM) over
// tiles_m * N/128 units; p.nstage from gemm_persistent_stages.
int gemm_persistent_stages(int BN);
cudaError_t launch_gemm_persistent(const CUtensorMap* mapA, const CUtensorMap* mapB, const GemmParams& p,
                                   int dtype, int grid, cudaStream_t s, bool pdl);

bool attn_supported(int head_dim, int group, int block_size);
int attn_max_grid(int dtype, int head_dim, int group, int batch);  // one full wave
cudaError_t launch_prefill(const PrefillParams& p, int dtype, int head_dim, int group,
                           cudaStream_t s, bool pdl);
// queue: launch the variant that may hand out units from p.sched (it does so when the rows hold
// at least kAttnQueueUnits units per CTA); false compiles the fixed deal alone.  Both give the
// same bits.
cudaError_t launch_attn(const AttnParams& p, int dtype, int head_dim, int group, int grid,
                        cudaStream_t s, bool pdl, bool queue);

cudaError_t launch_embed(const EmbedParams& p, int dtype, cudaStream_t s, bool pdl);
cudaError_t launch_argmax(const float* logits, int batch, int vocab, int32_t* out,
                          cudaStream_t s);
cudaError_t launch_kv_copy(const KvCopyParams& p, int sms, cudaStream_t s);

// Persistent step kernel (k_step.cu).
struct StepPlan {
  std::vector<long long> stream_off;  // [grid + 1] first chunk of each CTA's weight stream
  std::vector<long long> stream_lm;   // [grid] first LM-head chunk of each CTA's stream
};
// The CTAs' weight streams for the stages of p (n_tiles, kc, split, rot, n_layers); false when
// a split is outside 1..8 or a CTA would hold more split tiles than kStepMaxTilesPerCta.
bool build_step_plan(int grid, const StepParams& p, StepPlan* out);
size_t step_smem_bytes(int head_dim, int nslot);
cudaError_t step_configure(int dtype, int head_dim, size_t smem, int* blocks_per_sm);
cudaError_t launch_step(const StepParams& p, int dtype, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_step_pack(const PackDesc* desc, long long n, uint8_t* out, int head_dim,
                             cudaStream_t s);

// Record the text ns_last_error_message() returns on this thread.
void set_last_error(const char* msg);

}  // namespace ns

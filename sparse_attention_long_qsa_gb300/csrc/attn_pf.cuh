// The fp16 attention variant for calls with many tokens (attn_pf.cu): tiles
// of 64 cells, a cluster of two CTAs per (token, KV head), two CTAs per SM.
#pragma once

#include "qsa_internal.cuh"

namespace qsa {

// Whether the variant covers this call's shapes (fp16 K/V, several tiles per
// (token, KV head)); the caller takes it where one CTA per (token, KV head)
// is the cluster size its cost model gives.
bool attn_pf_eligible(const AttnArgs& a);
cudaError_t launch_attn_pf(const AttnArgs& a, unsigned* err, cudaStream_t stream);

}  // namespace qsa

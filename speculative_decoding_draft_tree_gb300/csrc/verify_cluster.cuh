// The one-launch form of spec_verify for small trees (internal to the library).
#pragma once

#include "common.cuh"
#include "kv_compact.cuh"

namespace spec {

struct ClusterVerifyArgs {
  const void* target;
  const void* draft;
  int64_t tld, dld;
  int32_t B, N, R, V, T_max, max_path;
  float tau, k2, inv_tau;   // k2 = log2(e) / tau
  int32_t probs, residual_rule;
  const int32_t* draft_row;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* node_offset;
  const int32_t* depth;
  const uint8_t* is_internal;
  const float* uniforms;
  int32_t* req_status;
  int32_t* out_tokens;
  int32_t* out_len;
  int32_t* path;
  int32_t* n_acc;
  int32_t* rejections;
  // KV compaction in the same launch (spec_verify_compact): compact != 0; cd.path, cd.n_acc,
  // cd.req_status and cd.max_path are the verification's own
  int32_t compact;
  CompactDev cd;
  // set at launch
  int32_t per_units;          // 8-element vocabulary units held by each CTA of a cluster
  int32_t t_slice, d_slice;   // shared-memory bytes of one target / draft row slice
  int32_t smem;               // dynamic shared memory of one CTA
};

// True when the call fits the one-launch form (the caller checks the sibling rule): trees of at
// most 32 nodes and, with 8 CTAs per request, one CTA's slices of a request's T_max target rows
// and T_max - 1 draft rows within 200 KiB.  tes / des: bytes per target / draft element.
bool verify_cluster_fits(const ClusterVerifyArgs& a, int tes, int des);

// Launches the call on `s` (cluster launch, programmatic dependent launch allowed) with the
// number of CTAs per request (1..8) that runs the batch in the fewest waves per unit of work.
// Returns cudaErrorNotSupported, having launched nothing, when the device holds no such
// cluster at once (the caller then takes the two-launch form).
cudaError_t launch_verify_cluster(const ClusterVerifyArgs& a, int tes, int des, cudaStream_t s);

}  // namespace spec

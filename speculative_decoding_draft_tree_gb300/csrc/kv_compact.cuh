// KV compaction's device arguments, shared by spec_kv_compact and the verification launch that
// compacts in the same kernel (internal to the library).
#pragma once

#include "common.cuh"

namespace spec {

struct CompactDev {
  char* k;
  char* v;
  int64_t layer_stride_bytes;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* path;
  const int32_t* n_acc;
  int32_t* req_status;
  int32_t* new_kv_len;
  int32_t* slot_map;
  int32_t* blocks_in_use;
  int32_t H_kv, row_bytes, bs, num_blocks, max_blocks, max_path, num_layers;
};

// Checks a spec_compact_params the way spec_kv_compact does and fills the device arguments.
spec_status_t make_compact_dev(const spec_compact_params* p, CompactDev* d);

}  // namespace spec

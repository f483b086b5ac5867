// mla_tc.h — the tcgen05 absorbed MLA decode for 128 query heads (mla_tc.cu), declared for the
// C-ABI layer (api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "launch.h"

namespace pkv {

// Requests one launch of the 128-head kernel holds (its shared memory goes to the rings and the P
// slots): a larger set takes consecutive launches over set positions [k * 256, (k + 1) * 256).
constexpr int kMlaTcSetChunk = 256;

// Workspace of the 128-head kernel: per cluster share, two partial slots of 128 rows x (512
// output dims + LSE) floats (the pieces of cut sequences), then one 64-bit merge record per
// share. p.ws_part points at the partials, p.ws_ctr at the records (mla_tc_meta_offset bytes in).
size_t mla_tc_workspace_bytes();
size_t mla_tc_meta_offset();
// Two launches: the cluster kernel, then the merge of cut sequences. tm as for launch_mla_decode.
cudaError_t launch_mla_tc(const DecodeParams& p, const CUtensorMap& tm, cudaStream_t stream, int* launches);

}  // namespace pkv

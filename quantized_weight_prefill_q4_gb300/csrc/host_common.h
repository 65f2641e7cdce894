// Host helpers shared by the TMA kernels' launchers (gemm_tc.cu, gemv_tc.cu):
// tensor-map encoding through the driver entry point, the programmatic-launch
// attribute and the SM count. Host only.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace apr {

// cuTensorMapEncodeTiled from the driver (once per process); nullptr, with a
// message in msg, if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn(char* msg, size_t msg_len);

// A 2-D tiled map over `outer` rows of `inner` elements, rows `row_bytes`
// apart, box box_inner x box_outer; elements outside the tensor read as zero.
bool make_map_2d(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                 uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swz, char* msg, size_t msg_len);

// Launch attribute that lets the kernel start before the preceding kernel of
// the stream has finished (it waits with griddepcontrol.wait where it must).
cudaLaunchAttribute pdl_attr();

// Streaming multiprocessors of the current device.
int num_sms();

}  // namespace apr

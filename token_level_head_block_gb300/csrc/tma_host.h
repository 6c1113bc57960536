// Host helpers shared by the launchers of the tensor-core kernels.
#pragma once

#include <cuda.h>

namespace mhla {

// cuTensorMapEncodeTiled for a bf16 tensor (driver entry point looked up once;
// interleave none, L2 promotion 256 B, out-of-bounds elements read as zero).
bool encode_tensor_map(CUtensorMap* m, int rank, void* base, const cuuint64_t* dims,
                       const cuuint64_t* strides_bytes, const cuuint32_t* box, CUtensorMapSwizzle swz);

// Streaming multiprocessors of the current device, 0 on error.
int device_sm_count();

}  // namespace mhla

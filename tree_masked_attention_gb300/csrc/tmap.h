// Host helper: TMA tensor maps through the driver entry point (no libcuda link).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tree {

// Tiled tensor map over a row-major tensor of `rank` dims (dims[0] innermost),
// strides_bytes[i] = byte stride of dim i+1, box = elements per dim, 128-byte swizzle
// when `swizzle128`. Out-of-range box elements read as zero. Returns TREE_OK or an
// error status (message recorded).
int make_tmap(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int rank, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);

}  // namespace tree

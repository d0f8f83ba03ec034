// The tree mask on the device: key j is visible to query i iff j <= i <= subtree_end[j]
// (Tree Training §3.2 "Attention Mask"; Trie packing, "Step 2 - Allow only ancestors and
// self"), evaluated for 32 consecutive keys at once from the padded subtree_end.
#pragma once
#include <cstdint>

namespace tree {

// Bit t set iff key jb + t is visible to query i (jb <= i <= subtree_end[jb + t]).
// endp is subtree_end padded with -1 to a multiple of 128 rows; jb a multiple of 32.
__device__ __forceinline__ uint32_t visible32(const int32_t* __restrict__ endp, int jb, int i) {
  const int4* e4 = reinterpret_cast<const int4*>(endp + jb);
  uint32_t bits = 0;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int4 e = __ldg(e4 + g);
    const int t = 4 * g;
    bits |= (static_cast<uint32_t>((jb + t <= i) && (i <= e.x)) |
             (static_cast<uint32_t>((jb + t + 1 <= i) && (i <= e.y)) << 1) |
             (static_cast<uint32_t>((jb + t + 2 <= i) && (i <= e.z)) << 2) |
             (static_cast<uint32_t>((jb + t + 3 <= i) && (i <= e.w)) << 3))
            << t;
  }
  return bits;
}

}  // namespace tree

// A token's k expert ids with every load issued before any is used.
#pragma once

#include <stdint.h>

namespace ep {

constexpr int kIdsMax = 8;  // ids held in registers

// Load the k ids of one row into ids[0..k) with one or two 16-byte loads
// when k is 4 or 8 and the row is 16-byte aligned; false otherwise (the
// caller then reads them one by one).
__device__ __forceinline__ bool load_ids(const int32_t* row, int k, int ids[kIdsMax]) {
  if ((k != 4 && k != 8) || (reinterpret_cast<uintptr_t>(row) & 15) != 0) return false;
  const int4 a = __ldg(reinterpret_cast<const int4*>(row));
  const int4 b = k == 8 ? __ldg(reinterpret_cast<const int4*>(row) + 1) : make_int4(-1, -1, -1, -1);
  ids[0] = a.x; ids[1] = a.y; ids[2] = a.z; ids[3] = a.w;
  ids[4] = b.x; ids[5] = b.y; ids[6] = b.z; ids[7] = b.w;
  return true;
}

}  // namespace ep

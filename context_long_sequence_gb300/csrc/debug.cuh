// debug.cuh -- bounds checks compiled into debug builds (-DCP_DEBUG).
//
// CP_IN_BOUNDS(cond, status) guards one global access or one TMA coordinate.
// Release builds: the macro is the constant `true` and `cond` is not
// evaluated, so the kernels are unchanged.  Debug builds: a false `cond`
// records {CP_ERR_DEVICE_BOUNDS, blockIdx.x, source line, file id} in
// status[0..3] (the first error since the last read wins) and the macro
// yields false; the caller then skips the access (TMA loads, whose
// out-of-range rows are filled with zeros by the hardware, are issued anyway
// so the transaction counts of their barriers stay whole).  Nothing traps;
// the host reads the record with cp_get_status_detail().
#pragma once
#include <cstdint>

#include "cp_attn.h"

namespace cpattn {

// File ids of the record.
enum : int32_t { kTuCpAttn = 1, kTuAttnFwd = 2, kTuAttnBwd = 3, kTuReshard = 4, kTuMerge = 5 };

inline __device__ bool debug_bounds_fail(int32_t* status, int line, int file) {
  if (status && atomicCAS(status, 0, CP_ERR_DEVICE_BOUNDS) == 0) {
    status[1] = static_cast<int32_t>(blockIdx.x);
    status[2] = line;
    status[3] = file;
    __threadfence();
  }
  return false;
}

}  // namespace cpattn

#ifdef CP_DEBUG
#define CP_IN_BOUNDS(cond, status) ((cond) || ::cpattn::debug_bounds_fail((status), __LINE__, CP_TU_ID))
#else
#define CP_IN_BOUNDS(cond, status) true
#endif

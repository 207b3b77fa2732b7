// Host-side preparation of one attention launch whose inputs are read in
// place, for entry points that keep the kernel's work list and per-head
// table in memory they own (mattn_noalloc.cu).  Defined in mattn_api.cpp.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "kernel_params.h"
#include "mattn.h"

namespace mattn {

// Everything one attention launch needs, prepared on the host: the
// parameter block with every field set except items, head_info and err
// (left null for the caller to point at its own device copies), and the
// host copies of the work list and of the per-head table (int32 [H][4]).
struct InPlaceLaunch {
  FwdParams p;
  std::vector<int2> items;
  std::vector<int32_t> head_info;
};

// Validates the call exactly as mattn_fwd does and prepares it, for inputs
// the kernel reads where they are: bf16, each head in raster order or in a
// column-major order whose grid has a multiple of 128 rows.  Inputs that
// need the reorder / convert pre-pass (fp32, explicit orders, other grids)
// give MATTN_ERR_UNSUPPORTED.  More than max_heads heads or max_items work
// items give MATTN_ERR_CAPACITY; both limits are checked before any CUDA
// call.  Then checks that the current device is sm_103 and encodes the
// TMA descriptors.  Allocates no device memory.  Sets the calling thread's
// last-error message on failure.
int prepare_in_place_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                            int d, int dtype, const mattn_mask_desc* desc, int max_heads, size_t max_items,
                            InPlaceLaunch* out);

// Sets the calling thread's last-error message (mattn_last_error) and
// returns code.
int report_error(int code, const char* fmt, ...);

}  // namespace mattn

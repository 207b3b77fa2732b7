// mattn_fwd_noalloc: the attention launch of mattn_fwd with the kernel's
// bookkeeping (error word, per-head table, work list) in a static device
// array of this file instead of memory allocated by the library, for
// callers that must not allocate device memory (include/mattn.h says who
// and why).  The attention kernel itself is the one mattn_fwd launches.
#include <cuda_runtime.h>

#include <mutex>

#include "kernel_params.h"
#include "launch_prep.h"
#include "mattn.h"

namespace mattn {
namespace {

// Layout of the static array (byte offsets; each part 256-byte aligned).
constexpr size_t kErrOffset = 0;      // uint32 error word
constexpr size_t kHeadOffset = 256;   // int32 [MATTN_NOALLOC_MAX_HEADS][4]
constexpr size_t kItemsOffset = kHeadOffset + 16 * (size_t)MATTN_NOALLOC_MAX_HEADS;  // int2 [MAX_ITEMS]
constexpr size_t kScratchBytes = MATTN_NOALLOC_SCRATCH_BYTES;
static_assert(kItemsOffset + 8 * (size_t)MATTN_NOALLOC_MAX_ITEMS == kScratchBytes, "scratch layout");
static_assert(kItemsOffset % 256 == 0, "work list alignment");

// One copy per device that loads the library, alive until the process ends.
// In host code this name is a host-side stand-in, not a device address: the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned char* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (the first call on each device).
int scratch_on_current_device(unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_error(MATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return report_error(MATTN_ERR_UNSUPPORTED, "device ordinal %d is beyond the %d devices supported here", dev,
                        kMaxDevices);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr)
      return report_error(MATTN_ERR_CUDA, "cudaGetSymbolAddress(scratch) on device %d: %s", dev,
                          cudaGetErrorString(e));
    g_scratch_addr[dev] = static_cast<unsigned char*>(ptr);
  }
  *out = g_scratch_addr[dev];
  return MATTN_OK;
}

#define MATTN_NOALLOC_CUDA(call, what)                                                                  \
  do {                                                                                                 \
    cudaError_t e_ = (call);                                                                           \
    if (e_ != cudaSuccess) return report_error(MATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e_)); \
  } while (0)

int fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                int dtype, const mattn_mask_desc* desc, cudaStream_t stream, uint32_t* wait_error_out) {
  InPlaceLaunch L;
  int rc = prepare_in_place_launch(q, k, v, o, lse, B, H, N, d, dtype, desc, MATTN_NOALLOC_MAX_HEADS,
                                   (size_t)MATTN_NOALLOC_MAX_ITEMS, &L);
  if (rc) return rc;
  // The work list and head table are uploaded from host vectors that live
  // only for this call; a graph would keep pointers to freed host memory, so
  // a stream under capture is refused before anything is recorded.
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  MATTN_NOALLOC_CUDA(cudaStreamIsCapturing(stream, &capture), "cudaStreamIsCapturing");
  if (capture != cudaStreamCaptureStatusNone)
    return report_error(MATTN_ERR_UNSUPPORTED,
                        "mattn_fwd_noalloc cannot run on a stream under graph capture (it uploads its work list "
                        "from host memory that lives only for the call)");
  unsigned char* scratch = nullptr;
  if ((rc = scratch_on_current_device(&scratch))) return rc;
  uint32_t* err = reinterpret_cast<uint32_t*>(scratch + kErrOffset);
  int32_t* head_info = reinterpret_cast<int32_t*>(scratch + kHeadOffset);
  int2* items = reinterpret_cast<int2*>(scratch + kItemsOffset);
  // Everything the kernel reads is rewritten, in stream order, before it
  // runs; the error word starts at zero.  The host vectors are pageable, so
  // each copy has taken its source before cudaMemcpyAsync returns.
  MATTN_NOALLOC_CUDA(cudaMemsetAsync(err, 0, sizeof(uint32_t), stream), "clear error word");
  MATTN_NOALLOC_CUDA(cudaMemcpyAsync(head_info, L.head_info.data(), L.head_info.size() * sizeof(int32_t),
                                     cudaMemcpyHostToDevice, stream),
                     "upload head table");
  if (!L.items.empty())
    MATTN_NOALLOC_CUDA(cudaMemcpyAsync(items, L.items.data(), L.items.size() * sizeof(int2), cudaMemcpyHostToDevice,
                                       stream),
                       "upload work list");
  L.p.items = items;
  L.p.head_info = head_info;
  L.p.err = err;
  MATTN_NOALLOC_CUDA(launch_attention(L.p, d, false, stream), "attention launch");
  if (wait_error_out) {
    uint32_t word = 0;
    MATTN_NOALLOC_CUDA(cudaStreamSynchronize(stream), "stream sync");
    MATTN_NOALLOC_CUDA(cudaMemcpy(&word, err, sizeof(word), cudaMemcpyDeviceToHost), "read error word");
    *wait_error_out = word;
    if (word & kErrBounds)
      return report_error(MATTN_ERR_BOUNDS, "a device bounds check failed (error word 0x%x)", word);
    if (word) return report_error(MATTN_ERR_TIMEOUT, "a device wait gave up (error word 0x%x)", word);
  }
  return MATTN_OK;
}

}  // namespace
}  // namespace mattn

extern "C" int mattn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                 int N, int d, int dtype, const mattn_mask_desc* desc, void* stream,
                                 uint32_t* wait_error_out) {
  std::lock_guard<std::mutex> lk(mattn::g_noalloc_mutex);
  return mattn::fwd_noalloc(q, k, v, o, lse, B, H, N, d, dtype, desc, static_cast<cudaStream_t>(stream),
                            wait_error_out);
}

// futr_decode_block_noalloc: the decode step with its scratch memory in a
// fixed-size array that lives in the library itself, for callers that cannot
// allocate device memory.
//
// Such callers include plugins hosted by a runtime that owns every device
// allocation, code running under a strict memory budget or a fixed
// allocator, and programs that must not call cudaMalloc at run time (its
// implicit synchronization and failure modes are unacceptable there).  They
// still own the inputs and outputs (x, the packed weights, the KV cache, pos,
// y); everything else the five kernels need -- intermediate activations,
// split-K and split-context partial sums, arrival counters and the error word
// -- comes from the array below.
#include <mutex>

#include "futr_internal.cuh"

namespace futr {
namespace host {
uint64_t workspace_bytes(const futr_shape& s, int max_batch, int capacity, int n_sm);
void describe_workspace(const futr_shape& s, int max_batch, int capacity, int n_sm, void* base, futr_ws* d);
int sm_count();
bool kv_valid(const futr_kv* kv);
futr_status check_decode_args(const void* blob, const futr_kv* kv, int layer, int batch, const futr_ws* ws);
futr_status launch_block(const uint16_t* x, const void* blob, const futr_kv* kv, int layer, int batch,
                         const int32_t* pos, uint16_t* y, const futr_ws* ws, cudaStream_t st);
}  // namespace host
}  // namespace futr

namespace {

// 48 MiB.  The scratch a call needs depends on the block shape, the batch and
// the SM count, not on the cache capacity: the 8B-shaped (hidden 4096) and
// 70B-shaped (hidden 8192) blocks need at most about 38 MB at batch 32 on a
// 152-SM device (mostly split-K partial sums).  Every device that loads the
// library keeps this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(48) << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (the name itself
// is only a host-side stand-in).  Resolved once per device.
futr_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FUTR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return FUTR_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FUTR_OK;
}

}  // namespace

extern "C" futr_status futr_decode_block_noalloc(const uint16_t* x, const void* blob, const futr_kv* kv,
                                                 int32_t layer, int32_t batch, const int32_t* pos, uint16_t* y,
                                                 void* stream) {
  if (!x || !pos || !y || x == y) return FUTR_ERR_INVALID_ARG;
  // the cache descriptor is checked before its shape sizes anything
  if (!futr::host::kv_valid(kv)) return FUTR_ERR_INVALID_ARG;
  if (batch < 1 || batch > futr::kMaxBatch) return FUTR_ERR_UNSUPPORTED;
  const int n_sm = futr::host::sm_count();
  if (n_sm <= 0) return FUTR_ERR_CUDA;
  const futr_shape& s = kv->shape;
  if (futr::host::workspace_bytes(s, batch, kv->capacity, n_sm) > kStaticScratchBytes)
    return FUTR_ERR_UNSUPPORTED;  // this shape/batch/capacity needs more than the fixed scratch
  void* base = nullptr;
  futr_status st = scratch_address(&base);
  if (st != FUTR_OK) return st;
  futr_ws ws;
  futr::host::describe_workspace(s, batch, kv->capacity, n_sm, base, &ws);
  st = futr::host::check_decode_args(blob, kv, layer, batch, &ws);
  if (st != FUTR_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // the arrival counters and the error region (error word and abort word)
  // must start at zero; the array keeps whatever the previous call left
  unsigned char* b = reinterpret_cast<unsigned char*>(base);
  if (cudaMemsetAsync(b + ws.off_cnt, 0, ws.cnt_words * 4, cs) != cudaSuccess) return FUTR_ERR_CUDA;
  if (cudaMemsetAsync(b + ws.off_err, 0, 16, cs) != cudaSuccess) return FUTR_ERR_CUDA;
  return futr::host::launch_block(x, blob, kv, layer, batch, pos, y, &ws, cs);
}

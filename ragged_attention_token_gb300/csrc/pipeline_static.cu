// rra_pipeline_static: the full pack -> attend -> unpack path for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is unavailable or forbidden
// -- inside a CUDA-graph capture region it does not own, in a plugin host
// whose memory is owned by someone else's pool (an inference server, a game
// or media engine), or in a real-time loop where an allocation's implicit
// device synchronisation would break the latency budget.  Such a caller can
// pass inputs and outputs but has no way to provide rra_pipeline's workspace.
//
// The scratch (cu_seqlens, pack indices and packed Q/K/V, laid out as
// rra_workspace_offsets() states) lives in one file-scope device array of a
// fixed size, which every GPU that loads this library holds until the
// process exits.  Host code cannot use the array's name as a device address
// (on the host it names a host-side stand-in), so the first call on each
// device looks the real address up with cudaGetSymbolAddress while that
// device is current, and later calls reuse it.
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace rra {
namespace {

static __device__ __align__(256) uint8_t g_static_scratch[RRA_STATIC_SCRATCH_BYTES];

constexpr int kMaxStaticDevices = 64;
uint8_t* g_scratch_ptr[kMaxStaticDevices] = {};
std::mutex g_scratch_mutex;

rra_status static_fail(rra_status s, const char* msg) {
  set_last_error_message(msg);
  return s;
}

// Device address of the scratch array on the current device (looked up once).
rra_status scratch_address(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_fail(RRA_ERR_CUDA, "rra_pipeline_static: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxStaticDevices)
    return static_fail(RRA_ERR_UNSUPPORTED, "rra_pipeline_static: device ordinal too large");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    uint8_t* ptr = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return static_fail(RRA_ERR_CUDA, "rra_pipeline_static: cudaGetSymbolAddress(scratch) failed");
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return RRA_OK;
}

}  // namespace
}  // namespace rra

extern "C" rra_status rra_pipeline_static(const uint8_t* keep, const void* q, const void* k, const void* v,
                                          int B, int N, int H, int d, float scale, rra_dtype in_dtype,
                                          void* out, rra_dtype out_dtype, void* stream) {
  using namespace rra;
  // Checks that rra_pack would only make after it has launched nothing yet,
  // so that a bad argument for the attention step enqueues no work at all.
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return static_fail(RRA_ERR_INVALID_ARG, "rra_pipeline_static: scale is not finite");
  if (out_dtype != RRA_F16 && out_dtype != RRA_BF16 && out_dtype != RRA_F32)
    return static_fail(RRA_ERR_INVALID_ARG, "rra_pipeline_static: output dtype invalid");
  if (out == nullptr) return static_fail(RRA_ERR_INVALID_ARG, "rra_pipeline_static: out is null");
  if ((reinterpret_cast<uintptr_t>(out) & 15u) != 0)
    return static_fail(RRA_ERR_MISALIGNED, "rra_pipeline_static: out not 16-byte aligned");
  const size_t need = rra_workspace_bytes(B, N, H, d, in_dtype);
  if (need == 0)
    return static_fail(RRA_ERR_UNSUPPORTED, "rra_pipeline_static: unsupported sizes or input dtype");
  if (need > static_cast<size_t>(RRA_STATIC_SCRATCH_BYTES))
    return static_fail(RRA_ERR_UNSUPPORTED,
                       "rra_pipeline_static: these sizes need more scratch than the 64 MiB static "
                       "maximum; call rra_pipeline with a workspace instead");
  uint8_t* ws = nullptr;
  rra_status st = scratch_address(&ws);
  if (st != RRA_OK) return st;
  size_t off[6];
  st = rra_workspace_offsets(B, N, H, d, in_dtype, off);
  if (st != RRA_OK) return st;
  int32_t* cu = reinterpret_cast<int32_t*>(ws + off[0]);
  int32_t* dst = reinterpret_cast<int32_t*>(ws + off[1]);
  int32_t* src = reinterpret_cast<int32_t*>(ws + off[2]);
  // Nothing in the scratch has to start at zero: the pack writes every
  // index and packed row that the attention step reads.
  st = rra_pack(keep, B, N, H, d, in_dtype, q, k, v, cu, dst, src, ws + off[3], ws + off[4], ws + off[5], out,
                out_dtype, stream);
  if (st != RRA_OK) return st;
  return rra_attend(ws + off[3], ws + off[4], ws + off[5], cu, B, N, H, d, scale, in_dtype, out, out_dtype, src,
                    N, stream);
}

// Unpack: scatter packed attention rows back to their padded positions.
//
// Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers",
// agents-report.net article, method overview bullet 3 (results written back
// to the original batch positions).  Positions whose token was pruned get
// +0 (the pages leave them unspecified; zero is this library's reading).
// The pipeline normally fuses this step into the attention epilogue plus
// the pack's zero fill; this standalone kernel serves callers that keep the
// packed output.
#include "common.cuh"

namespace rra {
namespace {

constexpr int THREADS = 256;

__global__ void __launch_bounds__(THREADS) unpack_kernel(const UnpackArgs a) {
  const long long total = static_cast<long long>(a.B) * a.N;
  const long long items = total * a.row_vecs;
  const long long cap = total;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (long long it = static_cast<long long>(blockIdx.x) * THREADS + threadIdx.x; it < items;
       it += static_cast<long long>(gridDim.x) * THREADS) {
    const long long g = it / a.row_vecs;
    const int c = static_cast<int>(it - g * a.row_vecs);
    const int t = __ldg(a.dst_idx + g);
    uint4 val = z;
    if (t >= 0) {
      if (t < cap) {
        val = __ldg(a.op + static_cast<size_t>(t) * a.row_vecs + c);
      } else if (c == 0) {
        record_error(a.err, RRA_DEVERR_INDEX_RANGE);
      }
    }
    a.out[static_cast<size_t>(g) * a.row_vecs + c] = val;
  }
}

}  // namespace

cudaError_t launch_unpack(const UnpackArgs& a, cudaStream_t stream) {
  const long long items = static_cast<long long>(a.B) * a.N * a.row_vecs;
  long long grid = (items + THREADS - 1) / THREADS;
  if (grid > 8 * 152 * 4) grid = 8 * 152 * 4;
  if (grid < 1) grid = 1;
  unpack_kernel<<<static_cast<unsigned>(grid), THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace rra

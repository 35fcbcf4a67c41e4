// The step before the path: an EViT-like pruning decision made on the
// device, so that progressive pruning needs no host round trip between
// layers.
//
// Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers",
// abstract (both revisions), which names EViT among the pruners the pipeline
// serves; the pages do not spell out its rule.  The reading taken here: an
// image's class token is its first kept token; a kept token's score is the
// class token's softmax attention weight on it, averaged over the heads; a
// pruning step keeps the class token and the top ceil(m * num / den) of the
// image's m other kept tokens by score, equal scores going to the lower
// position and a NaN score counting as -inf.
//
// cls_scores_kernel: one CTA per image.  Per head, each thread takes keys j
// with a stride: the 64-term dot product of the class query (staged in
// shared memory) with K row j in fp32, then a block max, exponentials in
// base 2, a block sum and the normalised weights accumulated per key in
// shared memory; the mean over heads goes to the key's original position.
//
// topk_keep_kernel: one CTA per image.  Every candidate's rank is the number
// of candidates that beat it (higher score, or equal score at a lower
// position), counted over the scores staged in shared memory; the candidate
// is kept iff its rank is below k.  O(N^2) comparisons per image, N <= 1024.
#include "common.cuh"

namespace rra {
namespace {

constexpr int PR_THREADS = 256;
constexpr int PR_WARPS = PR_THREADS / 32;
constexpr int PR_MAX_N = 1024;
constexpr int PR_HD = 64;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < PR_WARPS; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < PR_WARPS; ++w) r += red[w];
  return r;
}

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }

template <typename Tin>
__device__ __forceinline__ float dot_row(const float* q, const Tin* krow) {
  const uint4* k4 = reinterpret_cast<const uint4*>(krow);
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < PR_HD / 8; ++c) {
    const uint4 w = __ldg(k4 + c);
    const Tin* e = reinterpret_cast<const Tin*>(&w);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(q[8 * c + i], to_f(e[i]), acc);
  }
  return acc;
}

template <typename Tin>
__global__ void __launch_bounds__(PR_THREADS) cls_scores_kernel(const Tin* __restrict__ qp, const Tin* __restrict__ kp,
                                                                 const int32_t* __restrict__ cu,
                                                                 const int32_t* __restrict__ src, int B, int N, int H,
                                                                 float scale_log2, float* __restrict__ scores,
                                                                 int32_t* err) {
  __shared__ float acc[PR_MAX_N];
  __shared__ float w[PR_MAX_N];
  __shared__ float qrow[PR_HD];
  __shared__ float red[PR_WARPS];
  const int b = blockIdx.x;
  float* out = scores + static_cast<size_t>(b) * N;
  for (int j = threadIdx.x; j < N; j += PR_THREADS) out[j] = 0.f;
  const int s0 = __ldg(cu + b);
  const int n = __ldg(cu + b + 1) - s0;
  if (n <= 0 || n > N) {
    if (n < 0 && threadIdx.x == 0) record_error(err, RRA_DEVERR_SEQ_NEGATIVE);
    if (n > N && threadIdx.x == 0) record_error(err, RRA_DEVERR_SEQ_TOO_LONG);
    return;
  }
  for (int j = threadIdx.x; j < n; j += PR_THREADS) acc[j] = 0.f;
  for (int h = 0; h < H; ++h) {
    __syncthreads();   // the previous head is done with qrow and w
    if (threadIdx.x < PR_HD) qrow[threadIdx.x] = to_f(qp[(static_cast<size_t>(s0) * H + h) * PR_HD + threadIdx.x]);
    __syncthreads();
    float mx = -INFINITY;
    for (int j = threadIdx.x; j < n; j += PR_THREADS) {
      const float l = dot_row(qrow, kp + (static_cast<size_t>(s0 + j) * H + h) * PR_HD) * scale_log2;
      w[j] = l;
      mx = fmaxf(mx, l);
    }
    mx = block_max(mx, red);
    float sum = 0.f;
    for (int j = threadIdx.x; j < n; j += PR_THREADS) {
      const float p = exp2f(w[j] - mx);
      w[j] = p;
      sum += p;
    }
    sum = block_sum(sum, red);
    const float inv = 1.f / sum;
    for (int j = threadIdx.x; j < n; j += PR_THREADS) acc[j] += w[j] * inv;
  }
  __syncthreads();
  const float inv_h = 1.f / static_cast<float>(H);
  for (int j = threadIdx.x; j < n; j += PR_THREADS) {
    const long long pos = static_cast<long long>(__ldg(src + s0 + j)) - static_cast<long long>(b) * N;
    if (pos < 0 || pos >= N) {
      record_error(err, RRA_DEVERR_INDEX_RANGE);
      continue;
    }
    out[pos] = acc[j] * inv_h;
  }
}

__global__ void __launch_bounds__(PR_THREADS) topk_keep_kernel(const float* __restrict__ scores,
                                                                const uint8_t* __restrict__ keep_prev, int N,
                                                                int num, int den, uint8_t* __restrict__ keep_new) {
  __shared__ float s[PR_MAX_N];
  __shared__ unsigned char cand[PR_MAX_N];
  __shared__ int first;
  __shared__ float red[PR_WARPS];
  const int b = blockIdx.x;
  const uint8_t* row = keep_prev + static_cast<size_t>(b) * N;
  uint8_t* out = keep_new + static_cast<size_t>(b) * N;
  if (threadIdx.x == 0) first = N;
  __syncthreads();
  for (int j = threadIdx.x; j < N; j += PR_THREADS)
    if (row[j] != 0) atomicMin(&first, j);
  __syncthreads();
  const int c0 = first;   // the class token (N: the image keeps nothing)
  float m_local = 0.f;
  for (int j = threadIdx.x; j < N; j += PR_THREADS) {
    const bool c = row[j] != 0 && j != c0;
    cand[j] = c ? 1 : 0;
    const float v = scores[static_cast<size_t>(b) * N + j];
    s[j] = (v != v) ? -INFINITY : v;   // NaN counts as -inf
    m_local += c ? 1.f : 0.f;
  }
  const int m = static_cast<int>(block_sum(m_local, red));   // exact: at most 1024
  const long long k = (static_cast<long long>(m) * num + den - 1) / den;
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += PR_THREADS) {
    if (!cand[i]) {
      out[i] = (i == c0) ? 1 : 0;
      continue;
    }
    const float si = s[i];
    int rank = 0;
    for (int j = 0; j < N; ++j) {
      const float sj = s[j];
      rank += (cand[j] && (sj > si || (sj == si && j < i))) ? 1 : 0;
    }
    out[i] = (rank < k) ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_cls_scores(const void* qp, const void* kp, const int32_t* cu, const int32_t* src, int B, int N,
                              int H, float scale, rra_dtype in, float* scores, int32_t* err, cudaStream_t stream) {
  const float sl2 = scale * 1.4426950408889634f;
  if (in == RRA_BF16)
    cls_scores_kernel<__nv_bfloat16><<<B, PR_THREADS, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(qp), static_cast<const __nv_bfloat16*>(kp), cu, src, B, N, H, sl2, scores,
        err);
  else
    cls_scores_kernel<__half><<<B, PR_THREADS, 0, stream>>>(static_cast<const __half*>(qp),
                                                             static_cast<const __half*>(kp), cu, src, B, N, H, sl2,
                                                             scores, err);
  return cudaGetLastError();
}

cudaError_t launch_topk_keep(const float* scores, const uint8_t* keep_prev, int B, int N, int num, int den,
                             uint8_t* keep_new, cudaStream_t stream) {
  topk_keep_kernel<<<B, PR_THREADS, 0, stream>>>(scores, keep_prev, N, num, den, keep_new);
  return cudaGetLastError();
}

}  // namespace rra

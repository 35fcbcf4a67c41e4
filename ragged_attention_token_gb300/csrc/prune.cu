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
// topk_keep_kernel: one CTA per image.  Every candidate gets a 64-bit key
// (the score's bits ordered like the floats, above the complement of its
// position: keys are distinct, and a higher key is a higher score or an equal
// score at a lower position); its rank is the number of keys above its own,
// counted over the keys in shared memory, and it is kept iff the rank is
// below k.  O(N^2) comparisons per image, N <= 1024, one per instruction pair.
//
// prune_cls_kernel: the same decision with the scores taken from the
// attention kernel's class-token side output (weights per head, in packed
// order), and optionally the next layer's indices with it, so the pruning
// step costs one launch after the attention.
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

// Sort key of a candidate: the score's bits in an order that compares like
// the floats (a NaN counts as -inf) above the complement of its position, so
// that keys are distinct, a higher score wins and equal scores go to the lower
// position.  Non-candidates get key 0, below every candidate.
__device__ __forceinline__ unsigned long long cand_key(float v, int pos) {
  if (v != v) v = -INFINITY;
  const uint32_t b = __float_as_uint(v);
  const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(o) << 32) | static_cast<uint32_t>(~pos);
}

// Number of keys[0, n) above `k` (keys in shared memory; every thread of
// the warp reads the same key at a time, a broadcast).
__device__ __forceinline__ int keys_above(const unsigned long long* keys, int n, unsigned long long k) {
  int r0 = 0, r1 = 0;
  int j = 0;
  for (; j + 1 < n; j += 2) {
    r0 += keys[j] > k ? 1 : 0;
    r1 += keys[j + 1] > k ? 1 : 0;
  }
  if (j < n) r0 += keys[j] > k ? 1 : 0;
  return r0 + r1;
}

__device__ __forceinline__ int block_sum_int(int v, int* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int r = 0;
#pragma unroll
  for (int w = 0; w < PR_WARPS; ++w) r += red[w];
  return r;
}

__global__ void __launch_bounds__(PR_THREADS) topk_keep_kernel(const float* __restrict__ scores,
                                                                const uint8_t* __restrict__ keep_prev, int N,
                                                                int num, int den, uint8_t* __restrict__ keep_new) {
  __shared__ __align__(16) unsigned long long key[PR_MAX_N];
  __shared__ int first;
  __shared__ int red[PR_WARPS];
  asm volatile("griddepcontrol.wait;" ::: "memory");   // programmatic dependent of the kernel before it
  const int b = blockIdx.x;
  const uint8_t* row = keep_prev + static_cast<size_t>(b) * N;
  uint8_t* out = keep_new + static_cast<size_t>(b) * N;
  if (threadIdx.x == 0) first = N;
  __syncthreads();
  for (int j = threadIdx.x; j < N; j += PR_THREADS)
    if (row[j] != 0) atomicMin(&first, j);
  __syncthreads();
  const int c0 = first;   // the class token (N: the image keeps nothing)
  int m_local = 0;
  for (int j = threadIdx.x; j < N; j += PR_THREADS) {
    const bool c = row[j] != 0 && j != c0;
    key[j] = c ? cand_key(scores[static_cast<size_t>(b) * N + j], j) : 0ull;
    m_local += c ? 1 : 0;
  }
  const int m = block_sum_int(m_local, red);   // also orders the key writes before the reads below
  const long long k = (static_cast<long long>(m) * num + den - 1) / den;
  for (int i = threadIdx.x; i < N; i += PR_THREADS) {
    const unsigned long long ki = key[i];
    if (ki == 0ull) {
      out[i] = (i == c0) ? 1 : 0;
      continue;
    }
    out[i] = (keys_above(key, N, ki) < k) ? 1 : 0;
  }
}

// Rows image b keeps after a pruning step with fraction num/den: the class
// token and ceil((n-1) num / den) of the others; none for an empty image or
// an n outside [1, N] (recorded as an error by the image's own CTA).
__device__ __forceinline__ int kept_after(int n, int N, int num, int den) {
  if (n < 1 || n > N) return 0;
  return 1 + static_cast<int>((static_cast<long long>(n - 1) * num + den - 1) / den);
}

// The keep decision from the attention kernel's class-token side output:
// image b's score for its i-th row is the mean over heads of
// cls[b, h, i]; candidates are rows 1 .. n-1 (row 0 is the class token), in
// position order, so candidate c's rank is the number of candidates before
// it scoring at least as high plus those after it scoring higher (NaN scores
// read as -inf first).  One CTA per image.
// INDEX: also the next layer's indices, as the pack's index pass would
// write them for the new mask: the image's new offset is the sum of the
// kept counts of the images before it (every count follows from cu alone),
// a kept row's new packed row is that offset plus the kept rows before it,
// and rows[t] is its row in the previous packed layout (cu[b] + i).
template <int MAXN, bool INDEX>
__global__ void __launch_bounds__(PR_THREADS) prune_cls_kernel(const float* __restrict__ cls, int stride,
                                                                const int32_t* __restrict__ cu,
                                                                const int32_t* __restrict__ src, int B, int N, int H,
                                                                int num, int den, uint8_t* __restrict__ keep_new,
                                                                float* __restrict__ scores, int32_t* __restrict__ cu_new,
                                                                int32_t* __restrict__ dst_new,
                                                                int32_t* __restrict__ src_new,
                                                                int32_t* __restrict__ rows_new, int32_t* err) {
  __shared__ __align__(16) float cand[MAXN];
  __shared__ int red[PR_WARPS];
  // Launched as a programmatic dependent of the attention that writes cls:
  // nothing in global memory is touched before that kernel has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x;
  const size_t row0 = static_cast<size_t>(b) * N;
  for (int j = threadIdx.x; j < N; j += PR_THREADS) {
    if (keep_new != nullptr) keep_new[row0 + j] = 0;
    if (scores != nullptr) scores[row0 + j] = 0.f;
    if constexpr (INDEX) dst_new[row0 + j] = -1;
  }
  const int s0 = __ldg(cu + b);
  const int n = __ldg(cu + b + 1) - s0;
  int off = 0;
  if constexpr (INDEX) {
    int part = 0;
    for (int bb = threadIdx.x; bb < b; bb += PR_THREADS) part += kept_after(__ldg(cu + bb + 1) - __ldg(cu + bb), N, num, den);
    off = block_sum_int(part, red);
    if (threadIdx.x == 0) {
      cu_new[b] = off;
      if (b == B - 1) cu_new[B] = off + kept_after(n, N, num, den);
    }
  }
  if (n <= 0 || n > N) {
    if (n < 0 && threadIdx.x == 0) record_error(err, RRA_DEVERR_SEQ_NEGATIVE);
    if (n > N && threadIdx.x == 0) record_error(err, RRA_DEVERR_SEQ_TOO_LONG);
    return;
  }
  const float inv_h = 1.f / static_cast<float>(H);
  const float* img = cls + static_cast<size_t>(b) * H * stride;
  // Each thread keeps the scores and positions of its own rows.
  constexpr int PER = MAXN / PR_THREADS;
  float score[PER];
  int pos[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int i = threadIdx.x + r * PR_THREADS;
    score[r] = 0.f;
    pos[r] = -1;
    if (i < n) {
      float acc = 0.f;
      for (int h = 0; h < H; ++h) acc += __ldg(img + static_cast<size_t>(h) * stride + i);
      score[r] = acc * inv_h;
      const long long p = static_cast<long long>(__ldg(src + s0 + i)) - static_cast<long long>(b) * N;
      if (p < 0 || p >= N) record_error(err, RRA_DEVERR_INDEX_RANGE);
      else pos[r] = static_cast<int>(p);
      if (i > 0) cand[i - 1] = (score[r] != score[r]) ? -INFINITY : score[r];
    }
  }
  const int m = n - 1;
  const long long k = (static_cast<long long>(m) * num + den - 1) / den;
  __syncthreads();   // the candidates, and the filled rows, before the reads and writes below
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int running = 0;   // INDEX: kept rows in the slices before this one
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int i = threadIdx.x + r * PR_THREADS;
    bool kept = false;
    if (i < n) {
      kept = true;
      if (i > 0) {
        const int c = i - 1;
        const float x = cand[c];
        int r0 = 0, r1 = 0;
        int j = 0;
        for (; j + 1 < c; j += 2) {
          r0 += cand[j] >= x ? 1 : 0;
          r1 += cand[j + 1] >= x ? 1 : 0;
        }
        if (j < c) r0 += cand[j] >= x ? 1 : 0;
        for (j = c + 1; j + 1 < m; j += 2) {
          r0 += cand[j] > x ? 1 : 0;
          r1 += cand[j + 1] > x ? 1 : 0;
        }
        if (j < m) r0 += cand[j] > x ? 1 : 0;
        kept = r0 + r1 < k;
      }
      if (pos[r] >= 0) {
        if (keep_new != nullptr) keep_new[row0 + pos[r]] = kept ? 1 : 0;
        if (scores != nullptr) scores[row0 + pos[r]] = score[r];
      }
    }
    if constexpr (INDEX) {
      // Rank of this row among the image's kept rows: a block scan of the
      // slice's flags (warp ballots, then the warps' counts).
      const unsigned bal = __ballot_sync(0xffffffffu, kept);
      __syncthreads();   // red is free again
      if (lane == 0) red[warp] = __popc(bal);
      __syncthreads();
      int before = 0, total = 0;
#pragma unroll
      for (int w = 0; w < PR_WARPS; ++w) {
        const int cw = red[w];
        before += w < warp ? cw : 0;
        total += cw;
      }
      if (kept) {
        const int t = off + running + before + __popc(bal & ((1u << lane) - 1u));
        if (pos[r] >= 0) dst_new[row0 + pos[r]] = t;
        src_new[t] = static_cast<int32_t>(row0) + (pos[r] >= 0 ? pos[r] : 0);
        rows_new[t] = s0 + i;
      }
      running += total;
    }
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(PR_THREADS);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_keep_kernel, scores, keep_prev, N, num, den, keep_new);
}

cudaError_t launch_prune_cls(const float* cls, int stride, const int32_t* cu, const int32_t* src, int B, int N, int H,
                             int num, int den, uint8_t* keep_new, float* scores, int32_t* cu_new, int32_t* dst_new,
                             int32_t* src_new, int32_t* rows_new, int32_t* err, cudaStream_t stream) {
  // Programmatic stream serialisation: the launch overlaps the tail of the
  // attention kernel before it (which releases its dependents once every CTA
  // has issued its work); the kernel waits for that kernel's completion.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(PR_THREADS);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool index = cu_new != nullptr;
  if (N <= 256) {
    if (index)
      return cudaLaunchKernelEx(&cfg, prune_cls_kernel<256, true>, cls, stride, cu, src, B, N, H, num, den, keep_new,
                                scores, cu_new, dst_new, src_new, rows_new, err);
    return cudaLaunchKernelEx(&cfg, prune_cls_kernel<256, false>, cls, stride, cu, src, B, N, H, num, den, keep_new,
                              scores, cu_new, dst_new, src_new, rows_new, err);
  }
  if (index)
    return cudaLaunchKernelEx(&cfg, prune_cls_kernel<PR_MAX_N, true>, cls, stride, cu, src, B, N, H, num, den,
                              keep_new, scores, cu_new, dst_new, src_new, rows_new, err);
  return cudaLaunchKernelEx(&cfg, prune_cls_kernel<PR_MAX_N, false>, cls, stride, cu, src, B, N, H, num, den, keep_new,
                            scores, cu_new, dst_new, src_new, rows_new, err);
}

}  // namespace rra

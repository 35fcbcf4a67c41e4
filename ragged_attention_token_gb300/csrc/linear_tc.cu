// Packed (varlen) linear layer on the tensor cores: the rest of a ViT block
// (QKV projection, output projection, MLP) run on the compact buffer, so
// pruned tokens cost no multiplies there either.
//
// Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers",
// agents-report.net article, section "問題：填充與派遣的瓶頸" (problem): the
// padded layout wastes bandwidth and masked multiplies; here the layer's
// GEMM covers only the T = cu_seqlens[B] kept rows, T read on the device.
//
// c[t, :] = a[t, :] W^T (+ bias) for t < T.  a [cap, K] and W [N, K] (the
// nn.Linear layout) are both K-major, so one tcgen05.mma kind::f16 per 16-wide
// K step reads both straight from 128-byte-swizzled shared memory.
//
// One CTA per 128 x 128 output tile; a tile whose first row is past T
// returns at once; two CTAs share an SM, so one's epilogue overlaps the
// other's products.  Warp 0 streams 64-wide K chunks of the A and W tiles
// through a 3-stage TMA ring; warp 1 (which also owns the 128 TMEM columns
// of the fp32 accumulator) issues the MMAs from converged code with
// elect.sync and commits each stage back to the producer; warps 2-5 read the
// accumulator (each its TMEM lane quadrant), add the bias and store their
// rows.  Every wait is bounded; a CTA that gives up records
// RRA_DEVERR_WAIT_TIMEOUT, lets copies and products in flight land, frees
// its TMEM and returns.
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace rra {
namespace {

constexpr int LM = 128;                                  // output rows per tile (TMEM lanes)
constexpr int LN = 128;                                  // output columns per tile (TMEM columns)
constexpr int LK = 64;                                   // K per stage (one 128-byte swizzled row)
constexpr int L_STAGES = 3;                              // 96 KB ring: two CTAs per SM
constexpr int L_THREADS = 192;
constexpr uint32_t L_A_BYTES = LM * 128;
constexpr uint32_t L_W_BYTES = LN * 128;
constexpr uint32_t L_STAGE_BYTES = L_A_BYTES + L_W_BYTES;
constexpr uint32_t L_OFF_BAR = L_STAGES * L_STAGE_BYTES;
constexpr uint32_t L_B_FULL = 0;                         // [L_STAGES]
constexpr uint32_t L_B_EMPTY = 8 * L_STAGES;             // [L_STAGES]
constexpr uint32_t L_B_ACCUM = 16 * L_STAGES;
constexpr uint32_t L_W_TMEM = L_B_ACCUM + 8;
constexpr uint32_t L_W_ABORT = L_W_TMEM + 4;
constexpr uint32_t L_SMEM = L_OFF_BAR + 128 + 1024;      // + barriers; slack to align the base to 1024 B
constexpr uint32_t L_TMEM_COLS = LN;

struct LinearArgs {
  const int32_t* cu;     // cu_seqlens [B + 1]; T = cu[B]
  int B;
  int cap;               // rows of a and c
  int K, N;
  const float* bias;     // [N] or null
  void* c;               // [cap, N]
  int32_t* err;
};

template <typename Tout>
__device__ __forceinline__ void store_row32(Tout* dst, const float* v);
template <>
__device__ __forceinline__ void store_row32<float>(float* dst, const float* v) {
  float4* p = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}
template <typename T2>
__device__ __forceinline__ uint32_t pack_pair(float x, float y);
template <>
__device__ __forceinline__ uint32_t pack_pair<__nv_bfloat162>(float x, float y) {
  __nv_bfloat162 t = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&t);
}
template <>
__device__ __forceinline__ uint32_t pack_pair<__half2>(float x, float y) {
  __half2 t = __floats2half2_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&t);
}
template <typename T2>
__device__ __forceinline__ void store_row32_half(void* dst, const float* v) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    p[i] = make_uint4(pack_pair<T2>(v[8 * i], v[8 * i + 1]), pack_pair<T2>(v[8 * i + 2], v[8 * i + 3]),
                      pack_pair<T2>(v[8 * i + 4], v[8 * i + 5]), pack_pair<T2>(v[8 * i + 6], v[8 * i + 7]));
}
template <>
__device__ __forceinline__ void store_row32<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  store_row32_half<__nv_bfloat162>(dst, v);
}
template <>
__device__ __forceinline__ void store_row32<__half>(__half* dst, const float* v) {
  store_row32_half<__half2>(dst, v);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(L_THREADS, 2)
    linear_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
                     const LinearArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int n0 = blockIdx.x * LN, m0 = blockIdx.y * LM;
  const int T = __ldg(a.cu + a.B);
  if (T < 0 || T > a.cap) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) record_error(a.err, RRA_DEVERR_INDEX_RANGE);
    return;
  }
  if (m0 >= T) return;   // the whole tile is past the packed rows in use

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto s_a = [&](int s) { return base + s * L_STAGE_BYTES; };
  auto s_w = [&](int s) { return base + s * L_STAGE_BYTES + L_A_BYTES; };
  const uint32_t bars = base + L_OFF_BAR;
  auto bar_full = [&](int s) { return bars + L_B_FULL + 8 * s; };
  auto bar_empty = [&](int s) { return bars + L_B_EMPTY + 8 * s; };
  const uint32_t bar_accum = bars + L_B_ACCUM, abort_flag = bars + L_W_ABORT;
  const volatile uint32_t* tmem_ptr = reinterpret_cast<const volatile uint32_t*>(gbase + L_OFF_BAR + L_W_TMEM);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 1) {
    tmem_alloc(bars + L_W_TMEM, L_TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < L_STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_accum, 1);
    st_shared_u32(abort_flag, 0u);
    fence_barrier_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_w);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  const int kchunks = a.K / LK;
  bool bad = false;

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    for (int kc = 0; kc < kchunks; ++kc) {
      const int s = kc % L_STAGES;
      if (kc >= L_STAGES) bad |= !mbar_wait_or_abort(bar_empty(s), ((kc / L_STAGES) - 1) & 1, abort_flag);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      if (lane == 0) {
        mbar_expect_tx(bar_full(s), L_STAGE_BYTES);
        tma_load_2d(s_a(s), &map_a, kc * LK, m0, bar_full(s));   // rows past cap read as zeros
        tma_load_2d(s_w(s), &map_w, kc * LK, n0, bar_full(s));
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ products
    const uint32_t idesc = idesc_f16(IsBf16<Tin>::value, 0, LM, LN);
    for (int kc = 0; kc < kchunks; ++kc) {
      const int s = kc % L_STAGES;
      bad |= !mbar_wait_or_abort(bar_full(s), (kc / L_STAGES) & 1, abort_flag);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      tc_fence_after();
      const bool leader = elect_one();
#pragma unroll
      for (int kk = 0; kk < LK / 16; ++kk) {
        const uint64_t da = sdesc(s_a(s) + kk * 32, 16, 1024), dw = sdesc(s_w(s) + kk * 32, 16, 1024);
        if (leader) umma_f16(tmem, da, dw, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
      }
      if (leader) umma_commit(bar_empty(s));
    }
    if (!bad && elect_one()) umma_commit(bar_accum);
  } else {
    // ------------------------------------------------------------ epilogue
    bad |= !mbar_wait_or_abort(bar_accum, 0, abort_flag);
    bad = __any_sync(0xffffffffu, bad);
    if (!bad) {
      tc_fence_after();
      const int quad = warp & 3;                  // this warp's TMEM lane quadrant
      const int row = quad * 32 + lane;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      Tout* out = static_cast<Tout*>(a.c) + static_cast<size_t>(m0 + row) * a.N + n0;
#pragma unroll 1
      for (int g = 0; g < LN / 32; ++g) {
        float v[32];
        tmem_ld32(taddr + g * 32, v);
        if (a.bias != nullptr) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] += __ldg(a.bias + n0 + g * 32 + i);
        }
        if (m0 + row < T) store_row32<Tout>(out + g * 32, v);
      }
    }
  }
  if (bad && lane == 0) {
    st_shared_u32(abort_flag, 1u);
    record_error(a.err, RRA_DEVERR_WAIT_TIMEOUT);
  }

  // Teardown: after an abort, copies and products still in flight get a
  // bounded grace period (~1 ms) to land before the TMEM is released.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0 && ld_shared_volatile_u32(abort_flag) != 0u) {
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, L_TMEM_COLS);
  }
}

// 2-D map over a row-major [rows, K] matrix: box = 64 columns x 128 rows,
// 128-byte swizzle (the canonical K-major operand layout).
cudaError_t make_map_2d(CUtensorMap* map, PFN_cuTensorMapEncodeTiled_v12000 encode, const void* ptr, long long rows,
                        int K, bool bf16) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {LK, LM};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                      const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename Tin, typename Tout>
cudaError_t launch_linear_typed(const void* a_ptr, const void* w_ptr, const LinearArgs& a,
                                PFN_cuTensorMapEncodeTiled_v12000 encode, cudaStream_t stream) {
  auto kernel = linear_tc_kernel<Tin, Tout>;
  constexpr int kMaxDevices = 64;
  static bool attr_set[kMaxDevices] = {};
  static std::mutex m;
  int dev = 0;
  cudaError_t ed = cudaGetDevice(&dev);
  if (ed != cudaSuccess) return ed;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(m);
    if (!attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L_SMEM);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  CUtensorMap ma, mw;
  const bool bf16 = IsBf16<Tin>::value == 1;
  cudaError_t e = make_map_2d(&ma, encode, a_ptr, a.cap, a.K, bf16);
  if (e == cudaSuccess) e = make_map_2d(&mw, encode, w_ptr, a.N, a.K, bf16);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.N / LN), static_cast<unsigned>((a.cap + LM - 1) / LM));
  kernel<<<grid, L_THREADS, L_SMEM, stream>>>(ma, mw, a);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_linear_in(const void* a_ptr, const void* w_ptr, const LinearArgs& a, rra_dtype out,
                             PFN_cuTensorMapEncodeTiled_v12000 encode, cudaStream_t stream) {
  if (out == RRA_BF16) return launch_linear_typed<Tin, __nv_bfloat16>(a_ptr, w_ptr, a, encode, stream);
  if (out == RRA_F16) return launch_linear_typed<Tin, __half>(a_ptr, w_ptr, a, encode, stream);
  return launch_linear_typed<Tin, float>(a_ptr, w_ptr, a, encode, stream);
}

PFN_cuTensorMapEncodeTiled_v12000 linear_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

cudaError_t launch_linear_packed(const void* a_ptr, const void* w_ptr, const float* bias, const int32_t* cu, int B,
                                 int cap, int K, int N, rra_dtype in, void* c, rra_dtype out, int32_t* err,
                                 cudaStream_t stream) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = linear_encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  LinearArgs a{};
  a.cu = cu;
  a.B = B;
  a.cap = cap;
  a.K = K;
  a.N = N;
  a.bias = bias;
  a.c = c;
  a.err = err;
  if (in == RRA_BF16) return launch_linear_in<__nv_bfloat16>(a_ptr, w_ptr, a, out, encode, stream);
  return launch_linear_in<__half>(a_ptr, w_ptr, a, out, encode, stream);
}

}  // namespace rra

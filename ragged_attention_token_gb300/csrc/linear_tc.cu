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
// Persistent grid, one CTA per SM, each walking 128 x 256 output tiles
// (row-tile major, so CTAs running together share their A rows in L2; a
// short last round is split into 128-column tiles).  Warp 0 streams the
// 64-wide K chunks of the A and W tiles (16 + 32 KB) through a 4-stage TMA
// ring; warp 1 issues the 128 x 256 x 16 MMAs from converged code with
// elect.sync into one of two 256-column TMEM accumulators (all 512
// columns), so the next tile's products run while warps 2-9 drain the
// previous one (each warp a TMEM lane quadrant and half the columns: bias,
// conversion, then through 4 KB of shared memory per warp to coalesced
// stores of the rows below T; stored straight from the registers, one row
// per lane, the drain took longer than the products: 45 against 34 us on
// 12608 rows).  Every wait is bounded; a CTA that gives up records
// RRA_DEVERR_WAIT_TIMEOUT, lets copies and products in flight land, frees
// its TMEM and returns.
//
// What bounds it: per 128 x 256 x 16 product the SM's shared memory serves
// the MMA 12 KB of operands and takes 12 KB of TMA writes, about 190 bytes
// per cycle at the tensor rate, above what shared memory delivers -- so the
// products run at roughly two thirds of the tensor peak.  Sharing the W tile
// between two SMs by cluster multicast (less L2 traffic, the same shared
// memory traffic) and 256 x 256 tiles on one SM (the same bytes per product)
// measured no faster; pairing SMs on one product (the B operand split
// between them) is what lowers the per-SM traffic.
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace rra {
namespace {

constexpr int LM = 128;                                  // output rows per tile (TMEM lanes)
constexpr int LN = 256;                                  // output columns per tile (one accumulator)
constexpr int LK = 64;                                   // K per stage (one 128-byte swizzled row)
constexpr int L_STAGES = 4;                              // 192 KB ring: one CTA per SM
constexpr int L_EPI_WARPS = 8;                           // warps 2-9
constexpr int L_THREADS = 64 + 32 * L_EPI_WARPS;
constexpr uint32_t L_A_BYTES = LM * 128;
constexpr uint32_t L_W_BYTES = LN * 128;
constexpr uint32_t L_STAGE_BYTES = L_A_BYTES + L_W_BYTES;
constexpr uint32_t L_OFF_BAR = L_STAGES * L_STAGE_BYTES;
constexpr uint32_t L_B_FULL = 0;                         // [L_STAGES]
constexpr uint32_t L_B_EMPTY = 8 * L_STAGES;             // [L_STAGES]
constexpr uint32_t L_B_ACC_FULL = 16 * L_STAGES;         // [2] accumulator b complete
constexpr uint32_t L_B_ACC_EMPTY = L_B_ACC_FULL + 16;    // [2] accumulator b read out (one arrive per epilogue warp)
constexpr uint32_t L_W_TMEM = L_B_ACC_EMPTY + 16;
constexpr uint32_t L_W_ABORT = L_W_TMEM + 4;
// Output staging: per epilogue warp 32 rows x 128 bytes, rows swizzled in
// 16-byte chunks, so registers go in and coalesced row pieces come out
// without bank conflicts.
constexpr uint32_t L_OUT_BYTES = 32 * 128;
constexpr uint32_t L_OFF_OUT = L_OFF_BAR + 1024;
constexpr uint32_t L_SMEM = L_OFF_OUT + L_EPI_WARPS * L_OUT_BYTES + 1024;   // slack to align the base to 1024 B
constexpr uint32_t L_TMEM_COLS = 2 * LN;

struct LinearArgs {
  const int32_t* cu;     // cu_seqlens [B + 1]; T = cu[B]
  int B;
  int cap;               // rows of a and c
  int K, N;
  const float* bias;     // [N] or null
  void* c;               // [cap, N]
  int32_t* err;
};

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

// 16-byte chunk j of a 128-byte output row piece held as floats in v.
template <typename Tout>
__device__ __forceinline__ void pack_chunk(const float* v, int j, uint32_t (&w)[4]);
template <>
__device__ __forceinline__ void pack_chunk<float>(const float* v, int j, uint32_t (&w)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = __float_as_uint(v[4 * j + i]);
}
template <>
__device__ __forceinline__ void pack_chunk<__nv_bfloat16>(const float* v, int j, uint32_t (&w)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = pack_pair<__nv_bfloat162>(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
}
template <>
__device__ __forceinline__ void pack_chunk<__half>(const float* v, int j, uint32_t (&w)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = pack_pair<__half2>(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(L_THREADS, 1)
    linear_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
                     const __grid_constant__ CUtensorMap map_w_half, const LinearArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int T = __ldg(a.cu + a.B);
  if (T < 0 || T > a.cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(a.err, RRA_DEVERR_INDEX_RANGE);
    return;
  }
  // The CTA's tiles, 128 rows x 256 columns, row-tile major, CTA c taking
  // tiles c, c + G, c + 2G, ... (G = gridDim.x).  When the last round would
  // hold at most G/2 of them, its tiles are split into 128-column halves, so
  // the round takes about two thirds of the time of a full-width one (a
  // half-width tile moves more operand bytes per product).
  const int G = static_cast<int>(gridDim.x);
  const int n_wide = (a.N + LN - 1) / LN;
  const int mt = (T + LM - 1) / LM;
  const int wide_all = mt * n_wide;
  int wide = wide_all, narrow = 0;
  if (wide_all > G && 2 * (wide_all % G) <= G) {
    wide = wide_all - wide_all % G;
    narrow = 2 * (wide_all % G);
  }
  const int tiles = wide + narrow;
  if (static_cast<int>(blockIdx.x) >= tiles) return;   // nothing for this CTA (T read on the device)
  const int my_tiles = (tiles - static_cast<int>(blockIdx.x) + G - 1) / G;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto s_a = [&](int s) { return base + s * L_STAGE_BYTES; };
  auto s_w = [&](int s) { return base + s * L_STAGE_BYTES + L_A_BYTES; };
  const uint32_t bars = base + L_OFF_BAR;
  auto bar_full = [&](int s) { return bars + L_B_FULL + 8 * s; };
  auto bar_empty = [&](int s) { return bars + L_B_EMPTY + 8 * s; };
  auto bar_acc_full = [&](int b) { return bars + L_B_ACC_FULL + 8 * b; };
  auto bar_acc_empty = [&](int b) { return bars + L_B_ACC_EMPTY + 8 * b; };
  const uint32_t abort_flag = bars + L_W_ABORT;
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full(b), 1);
      mbar_init(bar_acc_empty(b), L_EPI_WARPS);
    }
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
  // Tile i of this CTA: origin and width (256, or 128 for a split tile of
  // the last round; a 128-column half past N is not a tile).
  auto tile_of = [&](int i, int& m0, int& n0, int& ln) {
    const int t = static_cast<int>(blockIdx.x) + i * G;
    if (t < wide) {
      m0 = (t / n_wide) * LM;
      n0 = (t % n_wide) * LN;
      ln = LN;
    } else {
      const int w = wide + ((t - wide) >> 1);
      m0 = (w / n_wide) * LM;
      n0 = (w % n_wide) * LN + ((t - wide) & 1) * (LN / 2);
      ln = LN / 2;
    }
  };
  if (warp == 0) {
    // ------------------------------------------------------------ loads
    uint32_t it = 0;   // K chunks issued so far (over all tiles)
    for (int i = 0; i < my_tiles && !bad; ++i) {
      int m0, n0, ln;
      tile_of(i, m0, n0, ln);
      const bool skip = n0 >= a.N;   // the half past N of a split tile: loads nothing, computes nothing
      for (int kc = 0; kc < kchunks; ++kc, ++it) {
        const int s = static_cast<int>(it % L_STAGES);
        if (it >= L_STAGES) bad |= !mbar_wait_or_abort(bar_empty(s), ((it / L_STAGES) - 1) & 1, abort_flag);
        bad = __any_sync(0xffffffffu, bad);
        if (bad) break;
        if (lane == 0) {
          mbar_expect_tx(bar_full(s), skip ? 0u : L_A_BYTES + static_cast<uint32_t>(ln) * 128u);
          if (!skip) {
            tma_load_2d(s_a(s), &map_a, kc * LK, m0, bar_full(s));   // rows past cap read as zeros
            // 256 rows of W, or 128: rows past N read as zeros
            tma_load_2d(s_w(s), ln == LN ? &map_w : &map_w_half, kc * LK, n0, bar_full(s));
          }
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ products
    uint32_t it = 0;
    for (int i = 0; i < my_tiles && !bad; ++i) {
      int m0, n0, ln;
      tile_of(i, m0, n0, ln);
      const uint32_t idesc = idesc_f16(IsBf16<Tin>::value, 0, LM, ln);
      const int b = i & 1;
      if (i >= 2) bad |= !mbar_wait_or_abort(bar_acc_empty(b), ((i >> 1) - 1) & 1, abort_flag);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      tc_fence_after();
      const uint32_t acc = tmem + static_cast<uint32_t>(b * LN);
      for (int kc = 0; kc < kchunks; ++kc, ++it) {
        const int s = static_cast<int>(it % L_STAGES);
        bad |= !mbar_wait_or_abort(bar_full(s), (it / L_STAGES) & 1, abort_flag);
        bad = __any_sync(0xffffffffu, bad);
        if (bad) break;
        tc_fence_after();
        const bool leader = elect_one();
        if (n0 < a.N) {
#pragma unroll
          for (int kk = 0; kk < LK / 16; ++kk) {
            const uint64_t da = sdesc(s_a(s) + kk * 32, 16, 1024), dw = sdesc(s_w(s) + kk * 32, 16, 1024);
            if (leader) umma_f16(acc, da, dw, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (leader) umma_commit(bar_empty(s));
      }
      if (bad) break;
      if (elect_one()) umma_commit(bar_acc_full(b));
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                   // this warp's TMEM lane quadrant
    const int half = (warp - 2) >> 2;            // and half of the tile's columns
    for (int i = 0; i < my_tiles; ++i) {
      const int b = i & 1;
      bad |= !mbar_wait_or_abort(bar_acc_full(b), (i >> 1) & 1, abort_flag);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      tc_fence_after();
      int m0, n0, ln;
      tile_of(i, m0, n0, ln);
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(b * LN);
      // Pieces of 128 bytes per row (64 columns of 16-bit output, 32 of
      // fp32): TMEM -> registers (+ bias) -> the warp's staging rows ->
      // four whole row pieces per store instruction, rows below T only.
      constexpr int CPP = 128 / static_cast<int>(sizeof(Tout));
      const uint32_t stg = base + L_OFF_OUT + static_cast<uint32_t>(warp - 2) * L_OUT_BYTES;
      uint8_t* cbytes = static_cast<uint8_t*>(a.c);
#pragma unroll 1
      for (int p = 0; p < ((ln / 2) + CPP - 1) / CPP; ++p) {
        const int col0 = half * (ln / 2) + p * CPP;
        if (n0 + col0 >= a.N) break;             // N a multiple of 128: whole pieces past N
        float v[CPP];
#pragma unroll
        for (int q = 0; q < CPP / 32; ++q) tmem_ld32(taddr + col0 + q * 32, v + q * 32);
        if (a.bias != nullptr) {
          // 16-byte loads (the bias is 16-byte aligned, n0 + col0 a multiple of 4), the same for every lane.
          const float4* b4 = reinterpret_cast<const float4*>(a.bias + n0 + col0);
#pragma unroll
          for (int j = 0; j < CPP / 4; ++j) {
            const float4 bb = __ldg(b4 + j);
            v[4 * j] += bb.x;
            v[4 * j + 1] += bb.y;
            v[4 * j + 2] += bb.z;
            v[4 * j + 3] += bb.w;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t w[4];
          pack_chunk<Tout>(v, j, w);
          st_shared_v4(stg + lane * 128 + ((j ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int rr = 4 * r + (lane >> 3), cc = lane & 7;
          const uint4 val = ld_shared_v4(stg + rr * 128 + ((cc ^ (rr & 7)) << 4));
          const int grow = m0 + quad * 32 + rr;
          if (grow < T)
            *reinterpret_cast<uint4*>(cbytes + (static_cast<size_t>(grow) * a.N + n0 + col0) * sizeof(Tout) + cc * 16) =
                val;
        }
        __syncwarp();                            // read back before the next piece is written
      }
      // This warp's share of accumulator b is in registers and stored: the
      // products of tile i + 2 may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc_empty(b));
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

// 2-D map over a row-major [rows, K] matrix: box = 64 columns x box_rows rows,
// 128-byte swizzle (the canonical K-major operand layout).
cudaError_t make_map_2d(CUtensorMap* map, PFN_cuTensorMapEncodeTiled_v12000 encode, const void* ptr, long long rows,
                        int K, bool bf16, uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {LK, box_rows};
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
  cudaError_t e = make_map_2d(&ma, encode, a_ptr, a.cap, a.K, bf16, LM);
  CUtensorMap mwh;
  if (e == cudaSuccess) e = make_map_2d(&mw, encode, w_ptr, a.N, a.K, bf16, LN);
  if (e == cudaSuccess) e = make_map_2d(&mwh, encode, w_ptr, a.N, a.K, bf16, LN / 2);
  if (e != cudaSuccess) return e;
  // One CTA per SM (the grid is capped by the tiles of all cap rows; CTAs
  // past the tiles of the T rows in use return at once).
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long max_tiles = 2LL * ((a.cap + LM - 1) / LM) * ((a.N + LN - 1) / LN);
  const int grid = static_cast<int>(max_tiles < sms ? max_tiles : sms);
  kernel<<<grid, L_THREADS, L_SMEM, stream>>>(ma, mw, mwh, a);
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

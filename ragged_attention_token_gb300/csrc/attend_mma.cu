// Bidirectional ragged attention on the packed buffers, warp-level tensor
// core version (mma.sync m16n8k16, fp32 accumulation).
//
// Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers",
// abstract (non-causal attention over pruned ViT sequences of at most 197 /
// 577 tokens) and the agents-report.net article, method overview bullet 2
// (attention computed directly on the compact buffer).
//
// One CTA = one (image b, head h, 64-query tile).  The grid is sized from the
// host-known bound max_seqlen; each CTA reads cu_seqlens on the device and
// returns at once when its tile starts past the image's length, so nothing is
// ever read back to the host.  Four warps own 16 query rows each.  K/V blocks
// of 64 keys stream through a two-stage cp.async ring in XOR-swizzled shared
// memory (16-byte chunk c of row r lives at chunk c ^ (r & 7), which makes the
// ldmatrix row reads conflict-free).  Softmax is the online (running max /
// running sum) form in base 2.  P enters the P.V product as two terms of the
// input type (round-to-nearest hi part plus the rounded remainder), because a
// single bf16 rounding of the weights alone costs up to ~2e-3 of output error
// at these lengths; with the split the weights carry ~16 significant bits.
// Rows and keys past the image's end are zero-filled on load and masked to
// -inf, so whatever memory holds there (even NaN) never reaches a kept output.
#include "common.cuh"

namespace rra {
namespace {

constexpr int BM = 64;        // query rows per CTA
constexpr int BN = 64;        // keys per block
constexpr int HD = 64;        // head dim
constexpr int THREADS = 128;  // 4 warps

template <typename T> struct IsBf16;
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };
template <> struct IsBf16<__half> { static constexpr bool value = false; };

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int n = pred ? 16 : 0;   // 0 source bytes = zero fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Splits two fp32 weights into hi + lo parts of the input type: hi is the
// round-to-nearest value, lo the rounded remainder, so hi + lo carries about
// 16 significant bits (bf16) instead of 8.
template <bool BF16>
__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    __nv_bfloat162 l = __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
  } else {
    __half2 h = __floats2half2_rn(x, y);
    __half2 l = __floats2half2_rn(x - __low2float(h), y - __high2float(h));
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
  }
}

// Byte offset of (row, 16-byte chunk) in a swizzled [rows][64] 2-byte tile.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Loads rows [r0, r0+64) of head h of one sequence (rows >= n zero-filled).
template <typename Tin>
__device__ __forceinline__ void load_tile(uint32_t dst, const Tin* base, int seq_start, int r0, int n,
                                          int H, int h) {
#pragma unroll
  for (int i = 0; i < (BM * 8) / THREADS; ++i) {
    const int id = threadIdx.x + i * THREADS;
    const int row = id >> 3, ch = id & 7;
    const bool ok = (r0 + row) < n;
    const Tin* src = ok ? base + (static_cast<size_t>(seq_start + r0 + row) * H + h) * HD + ch * 8 : base;
    cp_async16(dst + swz(row, ch), src, ok);
  }
}

template <typename Tout> struct OutVec;
template <> struct OutVec<float> { static constexpr int per16 = 4; };
template <> struct OutVec<__nv_bfloat16> { static constexpr int per16 = 8; };
template <> struct OutVec<__half> { static constexpr int per16 = 8; };

template <typename Tout>
__device__ __forceinline__ void store_pair(Tout* p, float x, float y);
template <>
__device__ __forceinline__ void store_pair<float>(float* p, float x, float y) {
  *reinterpret_cast<float2*>(p) = make_float2(x, y);
}
template <>
__device__ __forceinline__ void store_pair<__nv_bfloat16>(__nv_bfloat16* p, float x, float y) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x, y);
}
template <>
__device__ __forceinline__ void store_pair<__half>(__half* p, float x, float y) {
  *reinterpret_cast<__half2*>(p) = __floats2half2_rn(x, y);
}

// Returns whether the CTA stored output.
template <typename Tin, typename Tout, bool SCATTER>
__device__ __forceinline__ bool attend_mma_tile(const AttendArgs& a) {
  constexpr bool BF16 = IsBf16<Tin>::value;
  // Q tile, then two stages of (K block, V block); all 64 x 64 x 2 B, 1024-B aligned.
  __shared__ __align__(1024) uint8_t smem[BM * 128 + 2 * 2 * BN * 128];

  const int qtile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int seq_start = __ldg(a.cu_seqlens + b);
  const int n = __ldg(a.cu_seqlens + b + 1) - seq_start;
  if (n < 0) {
    if (qtile == 0 && h == 0 && threadIdx.x == 0) record_error(a.err, RRA_DEVERR_SEQ_NEGATIVE);
    return false;
  }
  if (n > a.max_seqlen) {
    if (qtile == 0 && h == 0 && threadIdx.x == 0) record_error(a.err, RRA_DEVERR_SEQ_TOO_LONG);
    return false;
  }
  const int m0 = qtile * BM;
  if (m0 >= n) return false;

  const Tin* qp = static_cast<const Tin*>(a.qp);
  const Tin* kp = static_cast<const Tin*>(a.kp);
  const Tin* vp = static_cast<const Tin*>(a.vp);
  const int H = a.H;

  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + BM * 128;
  auto sK = [&](int stage) { return sKV + stage * (2 * BN * 128); };
  auto sV = [&](int stage) { return sKV + stage * (2 * BN * 128) + BN * 128; };

  const int nblocks = (n + BN - 1) / BN;
  load_tile(sQ, qp, seq_start, m0, n, H, h);
  load_tile(sK(0), kp, seq_start, 0, n, H, h);
  load_tile(sV(0), vp, seq_start, 0, n, H, h);
  cp_async_commit();

  // Output row of each 16-byte vector this thread stores in the epilogue
  // (-1: past the image), looked up now so the epilogue does not wait on
  // the scatter indices.
  constexpr int VPR = HD / OutVec<Tout>::per16;   // 16-byte vectors per row
  constexpr int VECS = BM * VPR / THREADS;        // per thread
  static_assert(BM * VPR % THREADS == 0, "epilogue vectors must divide evenly over the threads");
  long long dst_rows[VECS];
#pragma unroll
  for (int k = 0; k < VECS; ++k) {
    const int i = m0 + (static_cast<int>(threadIdx.x) + k * THREADS) / VPR;
    long long r = -1;
    if (i < n) {
      r = static_cast<long long>(seq_start) + i;   // packed row
      if constexpr (SCATTER) {
        r = __ldg(a.src_idx + r);
        if (r < 0 || r >= static_cast<long long>(a.B) * a.N) {
          record_error(a.err, RRA_DEVERR_INDEX_RANGE);
          r = -1;
        }
      }
    }
    dst_rows[k] = r;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t qf[4][4];
  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) o[j][r] = 0.f;
  float row_max[2] = {-INFINITY, -INFINITY};
  float row_sum[2] = {0.f, 0.f};

  for (int kb = 0; kb < nblocks; ++kb) {
    const int stage = kb & 1;
    if (kb + 1 < nblocks) {
      load_tile(sK(stage ^ 1), kp, seq_start, (kb + 1) * BN, n, H, h);
      load_tile(sV(stage ^ 1), vp, seq_start, (kb + 1) * BN, n, H, h);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    if (kb == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int row = warp * 16 + (lane & 15);
        const int ch = kk * 2 + (lane >> 4);
        ldmatrix_x4(sQ + swz(row, ch), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }

    // S = Q K^T for this warp's 16 rows and the block's 64 keys.
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) s[j][r] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {   // pairs of 8-key n-tiles
        const int key = jp * 16 + ((lane >> 4) << 3) + (lane & 7);
        const int ch = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(sK(stage) + swz(key, ch), b0, b1, b2, b3);
        mma16816<BF16>(s[2 * jp], qf[kk], b0, b1);
        mma16816<BF16>(s[2 * jp + 1], qf[kk], b2, b3);
      }
    }

    // Scale into the log2 domain and mask keys past the sequence end.
    const int key0 = kb * BN;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int key = key0 + j * 8 + ((lane & 3) << 1) + (r & 1);
        s[j][r] = key < n ? s[j][r] * a.scale_log2 : -INFINITY;
      }
    }

    // Online softmax: rows lane/4 (regs 0,1) and lane/4 + 8 (regs 2,3).
    float new_max[2] = {row_max[0], row_max[1]};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      new_max[0] = fmaxf(new_max[0], fmaxf(s[j][0], s[j][1]));
      new_max[1] = fmaxf(new_max[1], fmaxf(s[j][2], s[j][3]));
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      new_max[x] = fmaxf(new_max[x], __shfl_xor_sync(0xffffffffu, new_max[x], 1));
      new_max[x] = fmaxf(new_max[x], __shfl_xor_sync(0xffffffffu, new_max[x], 2));
    }
    float corr[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      corr[x] = fast_exp2(row_max[x] - new_max[x]);   // 0 on the first block (-inf)
      row_max[x] = new_max[x];
      row_sum[x] *= corr[x];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j][0] *= corr[0];
      o[j][1] *= corr[0];
      o[j][2] *= corr[1];
      o[j][3] *= corr[1];
    }

    // P as hi + lo A fragments of the input type; O += P_hi V + P_lo V.
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {   // 16 keys per k-step
      uint32_t ph[4], pl[4];
      float p[8];
      p[0] = fast_exp2(s[2 * kk][0] - row_max[0]);
      p[1] = fast_exp2(s[2 * kk][1] - row_max[0]);
      p[2] = fast_exp2(s[2 * kk][2] - row_max[1]);
      p[3] = fast_exp2(s[2 * kk][3] - row_max[1]);
      p[4] = fast_exp2(s[2 * kk + 1][0] - row_max[0]);
      p[5] = fast_exp2(s[2 * kk + 1][1] - row_max[0]);
      p[6] = fast_exp2(s[2 * kk + 1][2] - row_max[1]);
      p[7] = fast_exp2(s[2 * kk + 1][3] - row_max[1]);
      row_sum[0] += (p[0] + p[1]) + (p[4] + p[5]);
      row_sum[1] += (p[2] + p[3]) + (p[6] + p[7]);
      split2<BF16>(p[0], p[1], ph[0], pl[0]);
      split2<BF16>(p[2], p[3], ph[1], pl[1]);
      split2<BF16>(p[4], p[5], ph[2], pl[2]);
      split2<BF16>(p[6], p[7], ph[3], pl[3]);
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {   // pairs of 8-wide d tiles
        const int key = kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int ch = dp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(sV(stage) + swz(key, ch), b0, b1, b2, b3);
        mma16816<BF16>(o[2 * dp], ph, b0, b1);
        mma16816<BF16>(o[2 * dp + 1], ph, b2, b3);
        mma16816<BF16>(o[2 * dp], pl, b0, b1);
        mma16816<BF16>(o[2 * dp + 1], pl, b2, b3);
      }
    }
    __syncthreads();   // this stage is refilled by the next iteration's prefetch
  }

  // Finish the row sums across the quad and normalise.
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    row_sum[x] += __shfl_xor_sync(0xffffffffu, row_sum[x], 1);
    row_sum[x] += __shfl_xor_sync(0xffffffffu, row_sum[x], 2);
  }
  const float inv0 = 1.f / row_sum[0];
  const float inv1 = 1.f / row_sum[1];

  // Stage the 64 x 64 output tile in shared memory (reusing the K/V ring),
  // then write whole rows with 16-byte stores.
  Tout* so = reinterpret_cast<Tout*>(smem + BM * 128);
  constexpr int OSTRIDE = HD + 16 / static_cast<int>(sizeof(Tout));   // padded row (elements)
  {
    const int r_lo = warp * 16 + (lane >> 2);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int col = j * 8 + ((lane & 3) << 1);
      store_pair<Tout>(so + r_lo * OSTRIDE + col, o[j][0] * inv0, o[j][1] * inv0);
      store_pair<Tout>(so + (r_lo + 8) * OSTRIDE + col, o[j][2] * inv1, o[j][3] * inv1);
    }
  }
  __syncthreads();
  Tout* out = static_cast<Tout*>(a.o);
#pragma unroll
  for (int k = 0; k < VECS; ++k) {
    if (dst_rows[k] < 0) continue;
    const int id = static_cast<int>(threadIdx.x) + k * THREADS;
    const int row = id / VPR, c = id - row * VPR;
    const uint4 val = *reinterpret_cast<const uint4*>(so + row * OSTRIDE + c * OutVec<Tout>::per16);
    uint4* gp = reinterpret_cast<uint4*>(out + (static_cast<size_t>(dst_rows[k]) * H + h) * HD) + c;
    *gp = val;
  }
  return true;
}

// One CTA per (query tile, head, image); CTAs whose tile lies past the
// image's length (or whose image has a bad length) return at once.
template <typename Tin, typename Tout, bool SCATTER>
__global__ void __launch_bounds__(THREADS) attend_mma_kernel(const AttendArgs a) {
  const bool wrote = attend_mma_tile<Tin, Tout, SCATTER>(a);
  if (a.done_count != nullptr) signal_done(a, wrote);
}

template <typename Tin, typename Tout>
cudaError_t launch_typed(const AttendArgs& a, cudaStream_t stream, uint32_t* ctas) {
  dim3 grid((a.max_seqlen + BM - 1) / BM, a.H, a.B);
  const uint32_t n = grid.x * grid.y * grid.z;
  AttendArgs b = a;
  if (b.done_count != nullptr) b.done_target += n;
  if (ctas != nullptr) *ctas = n;
  if (b.src_idx != nullptr)
    attend_mma_kernel<Tin, Tout, true><<<grid, THREADS, 0, stream>>>(b);
  else
    attend_mma_kernel<Tin, Tout, false><<<grid, THREADS, 0, stream>>>(b);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend(const AttendArgs& a, rra_dtype in, rra_dtype out, cudaStream_t stream, uint32_t* ctas) {
  if (in == RRA_BF16) {
    if (out == RRA_BF16) return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, stream, ctas);
    if (out == RRA_F16) return launch_typed<__nv_bfloat16, __half>(a, stream, ctas);
    return launch_typed<__nv_bfloat16, float>(a, stream, ctas);
  }
  if (out == RRA_BF16) return launch_typed<__half, __nv_bfloat16>(a, stream, ctas);
  if (out == RRA_F16) return launch_typed<__half, __half>(a, stream, ctas);
  return launch_typed<__half, float>(a, stream, ctas);
}

}  // namespace rra

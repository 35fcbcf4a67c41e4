// Bidirectional ragged attention for small grids (serving batches): one CTA
// of four warps per (image, head, tile of 128 query rows), tcgen05.mma with
// TMEM accumulators, no warp specialisation.
//
// Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers",
// abstract (non-causal attention over pruned ViT sequences; at serving batch
// sizes the call's latency, not its arithmetic, is what counts) and the
// agents-report.net article, method overview bullets 1-3 (pack, attention on
// the compact rows, results back at their original positions).
//
// When the grid has about one unit per SM, the warp-specialised kernel is
// one latency chain per CTA, and its hand-offs between the loading, MMA and
// softmax warps (each an mbarrier round trip) are most of that chain.  Here
// the same four warps do every step, separated by CTA barriers:
//   1. the image's length (cu_seqlens, or a ballot scan of its keep row in
//      the fused pipeline, which also lists the kept positions);
//   2. every thread copies 16-byte pieces of the Q tile and of all the
//      image's K and V rows (up to 256) into 128-byte-swizzled shared
//      memory with cp.async; rows past the image repeat its last row;
//   3. per 64-key chunk: one elected thread of warp 0 issues S = Q K^T
//      (M=128, N=chunk rounded up to 16, K=64) into TMEM columns 0..63; the
//      softmax of each query row by its thread (the warp-specialised
//      kernel's code: lazy reference, P written over S as hi + lo parts);
//      then O += P_hi V + P_lo V into columns 64..127;
//   4. the epilogue: O normalised, stored at the row's packed or padded
//      position; in the fused pipeline the unit that owns the image's
//      pruned rows (the first empty query tile, else the last tile) writes
//      +0 to this head's rows of them.
// Each MMA batch completes on one mbarrier that every thread waits on
// (bounded: a wait that runs out records RRA_DEVERR_WAIT_TIMEOUT and every
// thread of the CTA leaves together, after a short grace period for the
// copies and products in flight).
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "softmax_tc.cuh"
#include "tc_ptx.cuh"

namespace rra {
namespace {

constexpr int SBM = 128;                 // query rows per unit (= TMEM lanes)
constexpr int SBN = 64;                  // keys per chunk
constexpr int STHREADS = 128;
constexpr uint32_t STMEM_COLS = 128;     // S/P: columns [0, 64); O: [64, 128)
constexpr uint32_t STMEM_O = 64;
constexpr uint32_t SQ_BYTES = SBM * 128;
constexpr uint32_t S_MISC = 32;          // mbarrier, TMEM word, abort flag, length words

template <typename Tin, typename Tout, bool SCATTER, bool FUSED, bool LIMIT>
__global__ void __launch_bounds__(STHREADS)
    attend_small_kernel(const AttendArgs a, int qtiles, int kv_rows) {
  constexpr bool BF = IsBf16<Tin>::value == 1;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base, sK = base + SQ_BYTES, sV = sK + static_cast<uint32_t>(kv_rows) * 128u;
  const uint32_t misc = sV + static_cast<uint32_t>(kv_rows) * 128u;
  const uint32_t bar = misc, w_tmem = misc + 8, abort_flag = misc + 12, w_n = misc + 16, w_s0 = misc + 20;
  const uint32_t pos = misc + S_MISC;     // fused: kept positions (int16), then pruned ones from the back
  const volatile uint32_t* tmem_ptr = reinterpret_cast<const volatile uint32_t*>(gbase + (misc - base) + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = a.B * a.H;
  const int u = blockIdx.x;
  const int qt = u / BH, bh = u - (u / BH) * BH;
  const int h = bh % a.H, b = bh / a.H;
  const int q0 = qt * SBM;
  const long long wlimit = LIMIT ? a.wait_limit : WAIT_LIMIT_CYCLES;

  // Warp 0 allocates the TMEM while warp 1 initialises the barrier and
  // finds the image's rows (the first global reads, after the previous
  // kernel in the stream has completed), so the two latencies overlap.
  if (warp == 0) {
    tmem_alloc(w_tmem, STMEM_COLS);
    tmem_relinquish();
  } else if (warp == 1) {
    if (lane == 0) {
      mbar_init(bar, 1);
      st_shared_u32(abort_flag, 0u);
      fence_barrier_init();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // 1. The image's length and the start of its rows.
    if constexpr (FUSED) {
      // All the row's mask bytes are loaded before the first ballot (N <= 256:
      // eight per lane), so the scan waits for memory once.
      const unsigned lt = (1u << lane) - 1u;
      const uint8_t* krow = a.keep + static_cast<size_t>(b) * a.N;
      bool flag[ATTEND_SMALL_MAX_KEYS / 32];
#pragma unroll
      for (int r = 0; r < ATTEND_SMALL_MAX_KEYS / 32; ++r) {
        const int j = r * 32 + lane;
        flag[r] = (j < a.N) && (__ldg(krow + j) != 0);
      }
      int cnt = 0;
#pragma unroll
      for (int r = 0; r < ATTEND_SMALL_MAX_KEYS / 32; ++r) {
        const int j = r * 32 + lane;
        const unsigned m = __ballot_sync(0xffffffffu, flag[r]);
        if (flag[r]) st_shared_u16(pos + 2u * static_cast<uint32_t>(cnt + __popc(m & lt)), static_cast<uint32_t>(j));
        cnt += __popc(m);
      }
      if (lane == 0) {
        st_shared_u32(w_n, static_cast<uint32_t>(cnt));
        st_shared_u32(w_s0, 0u);
      }
    } else {
      if (lane == 0) {
        int s0 = __ldg(a.cu_seqlens + b);
        int n = __ldg(a.cu_seqlens + b + 1) - s0;
        if (n < 0 || n > a.max_seqlen) {
          if (qt == 0 && h == 0) record_error(a.err, n < 0 ? RRA_DEVERR_SEQ_NEGATIVE : RRA_DEVERR_SEQ_TOO_LONG);
          n = 0;
        } else if (s0 < 0 || static_cast<long long>(s0) + n > static_cast<long long>(a.B) * a.max_seqlen) {
          if (qt == 0 && h == 0) record_error(a.err, RRA_DEVERR_INDEX_RANGE);
          n = 0;
        }
        st_shared_u32(w_n, static_cast<uint32_t>(n));
        st_shared_u32(w_s0, static_cast<uint32_t>(s0));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  // Every thread's global accesses come after the previous kernel has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = static_cast<int>(ld_shared_u32(w_n));
  const int s0 = static_cast<int>(ld_shared_u32(w_s0));
  const int rows_q = min(SBM, n - q0);
  bool bad = false;

  if (rows_q > 0) {
    // 2. Q tile, then every K and V row of the image (padded to 16 rows).
    const uint8_t* const qg = static_cast<const uint8_t*>(a.qp);
    const uint8_t* const kg = static_cast<const uint8_t*>(a.kp);
    const uint8_t* const vg = static_cast<const uint8_t*>(a.vp);
    auto row_off = [&](int t) -> size_t {
      size_t row;
      if constexpr (FUSED) row = static_cast<size_t>(b) * a.N + static_cast<size_t>(ld_shared_u16(pos + 2u * t));
      else row = static_cast<size_t>(s0 + t);
      return (row * a.H + h) * (HD * 2);
    };
    for (int p = tid; p < rows_q * 8; p += STHREADS) {
      const int r = p >> 3, ch = p & 7;
      cp_async16(sQ + swz128(r, ch), qg + row_off(q0 + r) + ch * 16);
    }
    const int npad = (n + 15) & ~15;
    for (int p = tid; p < npad * 8; p += STHREADS) {
      const int r = p >> 3, ch = p & 7;
      const size_t off = row_off(r < n ? r : n - 1) + ch * 16;
      cp_async16(sK + swz128(r, ch), kg + off);
      cp_async16(sV + swz128(r, ch), vg + off);
    }
    // Where this thread's row goes (element offset of its output row), or
    // -1; looked up while the copies are in flight, so the scatter index's
    // load does not add a round trip before the first product.
    long long out_elem = -1;
    {
      const int i = q0 + tid;
      if (i < n) {
        long long dst_row;
        if constexpr (FUSED) {
          dst_row = static_cast<long long>(b) * a.N + ld_shared_u16(pos + 2u * static_cast<uint32_t>(i));
        } else {
          dst_row = static_cast<long long>(s0) + i;
          if constexpr (SCATTER) {
            dst_row = __ldg(a.src_idx + dst_row);
            if (dst_row < 0 || dst_row >= static_cast<long long>(a.B) * a.N) {
              record_error(a.err, RRA_DEVERR_INDEX_RANGE);
              dst_row = -1;
            }
          }
        }
        out_elem = dst_row < 0 ? -1 : (dst_row * a.H + h) * HD;
      }
    }

    asm volatile("cp.async.wait_all;" ::: "memory");
    fence_proxy_async();   // the copies (generic proxy) before the products read them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // 3. Per chunk: S, softmax, P.V.
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS_row = tmem + lane_off, tO_row = tmem + STMEM_O + lane_off;
    const bool rows_here = warp * 32 < rows_q;   // warp-uniform
    const float c2 = a.scale_log2;
    const uint32_t idesc_pv = idesc_f16(BF ? 1u : 0u, 1, SBM, HD);
    float m_run = 0.f, l_run = 0.f;
    uint32_t ph = 0;
    const int nch = (n + SBN - 1) / SBN;
    for (int c = 0; c < nch && !bad; ++c) {
      const int n_c = min(SBN, n - c * SBN);
      const int nk16 = (n_c + 15) & ~15;
      if (warp == 0) {
        tc_fence_after();
        const uint32_t idesc_s = idesc_f16(BF ? 1u : 0u, 0, SBM, nk16);
        const bool leader = elect_one();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t da = sdesc(sQ + kk * 32, 16, 1024);
          const uint64_t db = sdesc(sK + c * SBN * 128 + kk * 32, 16, 1024);
          if (leader) umma_f16(tmem, da, db, idesc_s, kk > 0 ? 1u : 0u);
        }
        if (leader) umma_commit(bar);
        __syncwarp();
      }
      // Each thread waits for S on its own: no CTA barrier here (the next
      // completion on the barrier, P.V's, needs every thread past the one
      // below first, so no thread can miss this phase).
      bad |= !mbar_wait_or_abort(bar, ph, abort_flag, wlimit);
      bad = __any_sync(0xffffffffu, bad);   // warp-uniform: the softmax and TMEM loads are warp-wide
      ph ^= 1;
      tc_fence_after();
      if (rows_here && !bad) softmax_chunk64<BF>(tS_row, tO_row, nk16, n_c, c, tid < rows_q, c2, m_run, l_run);
      tc_fence_before();
      bad = __syncthreads_or(bad) != 0;   // every P written (and the CTA agrees on giving up)
      if (bad) break;
      if (warp == 0) {
        tc_fence_after();
        const bool leader = elect_one();
        for (int kk = 0; kk < nk16 / 16; ++kk) {
          const uint64_t db = sdesc(sV + c * SBN * 128 + kk * 2048, 8192, 1024);
          if (leader) umma_f16_tmem_a(tmem + STMEM_O, tmem + kk * 16, db, idesc_pv, (kk > 0 || c > 0) ? 1u : 0u);
        }
        for (int kk = 0; kk < nk16 / 16; ++kk) {
          const uint64_t db = sdesc(sV + c * SBN * 128 + kk * 2048, 8192, 1024);
          if (leader) umma_f16_tmem_a(tmem + STMEM_O, tmem + kk * 16 + 8, db, idesc_pv, 1u);
        }
        if (leader) umma_commit(bar);
        __syncwarp();
      }
      bad |= !mbar_wait_or_abort(bar, ph, abort_flag, wlimit);
      bad = __any_sync(0xffffffffu, bad);
      ph ^= 1;
      // Before the next chunk's S completes on the same barrier every thread
      // must have seen this phase (else its parity test would skip ahead).
      // (Skipped after the last chunk, the pipeline ran 2 % faster and the
      // packed-input attention 5 % slower.)
      bad = __syncthreads_or(bad) != 0;
      tc_fence_after();
    }

    // 4. Epilogue.
    if (!bad && rows_here) {
      const float inv = 1.f / l_run;
      Tout* out = static_cast<Tout*>(a.o) + (out_elem < 0 ? 0 : out_elem);
#pragma unroll
      for (int g = 0; g < HD / 16; ++g) {
        float o[16];
        tmem_ld16(tO_row + g * 16, o);
        if (out_elem >= 0) store16<Tout>(out + g * 16, o, inv);
      }
    }
    if constexpr (FUSED) {
      if (!bad && warp == 0 && qt == qtiles - 1) zero_pruned_rows<Tout>(a, b, h, lane);   // every tile has rows
    }
  } else if constexpr (FUSED) {
    // The image's first empty query tile owns this head's pruned rows.
    if (warp == 0 && q0 - SBM < n) zero_pruned_rows<Tout>(a, b, h, lane);
  }

  // Host completion word (rra_attend_wait): every output store of the CTA is
  // issued, so the host may see the count move before the teardown below.
  if constexpr (!FUSED) {
    if (a.done_count != nullptr) signal_done(a);
  }
  // Teardown (after an abort, a bounded grace period for copies and products
  // still in flight before the TMEM is released).
  tc_fence_before();
  if (__syncthreads_or(bad) && tid == 0) {
    st_shared_u32(abort_flag, 1u);
    record_error(a.err, RRA_DEVERR_WAIT_TIMEOUT);
  }
  __syncthreads();
  if (warp == 0) {
    if (lane == 0 && ld_shared_volatile_u32(abort_flag) != 0u) {
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, STMEM_COLS);
  }
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

constexpr int kMaxDevSmall = 64;

template <typename Tin, typename Tout, bool SCATTER, bool FUSED, bool LIMIT>
cudaError_t launch_small_typed(const AttendArgs& a, cudaStream_t stream, uint32_t* ctas) {
  auto kernel = attend_small_kernel<Tin, Tout, SCATTER, FUSED, LIMIT>;
  constexpr uint32_t kMaxSmem = 1024 + SQ_BYTES + 2u * ATTEND_SMALL_MAX_KEYS * 128u + S_MISC + 2u * 1024u;
  static bool attr_set[kMaxDevSmall] = {};
  static std::mutex m;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevSmall) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(m);
    if (!attr_set[dev]) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxSmem));
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  const int kv_rows = (a.max_seqlen + 31) & ~31;      // K and V rows held per unit (>= the padded length)
  const uint32_t smem = 1024 + SQ_BYTES + 2u * static_cast<uint32_t>(kv_rows) * 128u + S_MISC +
                        (FUSED ? static_cast<uint32_t>((2 * a.N + 15) & ~15) : 0u);
  const int qtiles = (a.max_seqlen + SBM - 1) / SBM;
  const long long units = static_cast<long long>(a.B) * a.H * qtiles;
  AttendArgs b = a;
  if (b.done_count != nullptr) b.done_target += static_cast<uint32_t>(units);
  if (ctas != nullptr) *ctas = static_cast<uint32_t>(units);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units));
  cfg.blockDim = dim3(STHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, b, qtiles, kv_rows);
}

template <typename Tin, typename Tout, bool FUSED>
cudaError_t launch_small_lim(const AttendArgs& a, cudaStream_t stream, uint32_t* ctas) {
  const bool scatter = !FUSED && a.src_idx != nullptr;
  if (a.wait_limit > 0) {
    if (scatter) return launch_small_typed<Tin, Tout, true, FUSED, true>(a, stream, ctas);
    return launch_small_typed<Tin, Tout, false, FUSED, true>(a, stream, ctas);
  }
  if (scatter) return launch_small_typed<Tin, Tout, true, FUSED, false>(a, stream, ctas);
  return launch_small_typed<Tin, Tout, false, FUSED, false>(a, stream, ctas);
}

template <typename Tin, bool FUSED>
cudaError_t launch_small_in(const AttendArgs& a, rra_dtype out, cudaStream_t stream, uint32_t* ctas) {
  if (out == RRA_BF16) return launch_small_lim<Tin, __nv_bfloat16, FUSED>(a, stream, ctas);
  if (out == RRA_F16) return launch_small_lim<Tin, __half, FUSED>(a, stream, ctas);
  return launch_small_lim<Tin, float, FUSED>(a, stream, ctas);
}

}  // namespace

cudaError_t launch_attend_small(const AttendArgs& a, rra_dtype in, rra_dtype out, bool fused, cudaStream_t stream,
                                uint32_t* ctas) {
  if (a.max_seqlen < 1 || a.max_seqlen > ATTEND_SMALL_MAX_KEYS) return cudaErrorInvalidValue;
  if (fused && (a.keep == nullptr || a.N != a.max_seqlen)) return cudaErrorInvalidValue;
  if (fused) {
    if (in == RRA_BF16) return launch_small_in<__nv_bfloat16, true>(a, out, stream, ctas);
    return launch_small_in<__half, true>(a, out, stream, ctas);
  }
  if (in == RRA_BF16) return launch_small_in<__nv_bfloat16, false>(a, out, stream, ctas);
  return launch_small_in<__half, false>(a, out, stream, ctas);
}

}  // namespace rra

// Bidirectional ragged attention on the packed buffers, sm_103a tensor-core
// version: TMA tile loads, tcgen05.mma with TMEM accumulators.
//
// Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers",
// abstract (non-causal attention over pruned ViT sequences of at most 197 /
// 577 tokens) and the agents-report.net article, method overview bullet 2
// (attention computed directly on the compact buffer).
//
// Work unit = (image b, head h, tile of 128 query rows).  Persistent CTAs of
// 128 threads (four per SM) walk the units with a grid stride; a unit whose
// tile starts past the image's length (read from cu_seqlens on the device)
// costs two loads and is skipped.  Per unit, keys stream in chunks of 64:
//
//   TMA   Q tile (once) and the chunk's K and V rows -> shared memory, in
//         32-row boxes of the packed [T, H, 64] tensor with the 128-byte
//         swizzle, so at most 31 rows past the image are fetched;
//   MMA   S = Q K^T (M=128, N=chunk rounded up to 16, K=64) -> TMEM cols 0..63;
//   SIMT  thread r owns query row r (TMEM lane r): it reads its S row, takes
//         the softmax max in base 2, and writes P as two bf16/fp16 parts
//         (hi = round(p), lo = round(p - hi)) back over S in TMEM;
//   MMA   O += P_hi V + P_lo V (M=128, N=64, K=chunk), A read from TMEM,
//         O accumulating in TMEM cols 64..127 across the unit's chunks.
//
// The softmax is lazily rescaled: exponentials use a per-row reference max
// that only moves (rescaling O in TMEM) when a chunk's max exceeds it by
// more than 8 in the log2 domain (bf16: a single pass against the running
// reference, redone exactly only when a row's chunk sum exceeds 2^32).
// The next item's K/V loads are issued before the current item computes (two
// stages) and the next unit's Q right after the current unit's last S product.
//
// P is split because one bf16 rounding of the weights alone leaves up to
// ~2e-3 of output error at these lengths; hi + lo carries ~16 bits.  Keys
// past the image's end are masked (p = 0) and the V rows the MMA reads past
// the end are zeroed in shared memory, so whatever the buffer holds there
// (even NaN) never reaches a kept output.  Every mbarrier wait is bounded
// by a clock-cycle limit: on expiry the CTA records RRA_DEVERR_WAIT_TIMEOUT,
// waits (bounded) for its own copies, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace rra {
namespace {

constexpr int BM = 128;        // query rows per unit (= TMEM lanes)
constexpr int BN = 64;         // keys per chunk
constexpr int HD = 64;         // head dim
constexpr int CONSUMERS = 128;   // warps 0-3: MMA issue (thread 0) and softmax, one query row each
constexpr int THREADS = CONSUMERS + 32;   // warp 4: TMA producer
constexpr int BOX = 32;        // rows per TMA box (packed inputs)
constexpr int CTAS_PER_SM = 4;
constexpr int STAGES = 2;      // K/V chunk ring

constexpr uint32_t Q_BYTES = BM * 128;                 // 128 rows x 128 B
constexpr uint32_t KV_BYTES = BN * 128;                //  64 rows x 128 B
constexpr uint32_t OFF_Q = 0;                          // one Q tile
constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;            // K[STAGES]
constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;  // V[STAGES]
constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
// mbarriers: full[2] +0/+8, empty[2] +16/+24, qempty +32, mma +40; TMEM slot +48;
// abort flag +52; redo flags +56/+60; item descriptors (2 x 48 B) +64; then,
// for the fused pipeline, POS_SLOTS lists of kept positions (int16, N each).
constexpr uint32_t DESC_BYTES = 48;
constexpr uint32_t OFF_DESC = OFF_BAR + 64;
constexpr uint32_t OFF_POS = OFF_DESC + STAGES * DESC_BYTES;
constexpr int POS_SLOTS = 3;
constexpr uint32_t SMEM_ALLOC = OFF_POS + 1024;        // + position lists; slack to align the base to 1024 B

enum { MODE_PACKED = 0, MODE_GATHER = 1, MODE_FUSED = 2 };
constexpr uint32_t TMEM_COLS = 128;                    // S/P: cols [0,64), O: cols [64,128)
constexpr uint32_t WAIT_SUSPEND_NS = 20000;            // try_wait suspend hint
constexpr long long WAIT_LIMIT_CYCLES = 2000000000LL;  // ~1 s at 2 GHz

template <typename T> struct IsBf16;
template <> struct IsBf16<__nv_bfloat16> { static constexpr uint32_t value = 1; };
template <> struct IsBf16<__half> { static constexpr uint32_t value = 0; };

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ mbarrier / TMA

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(WAIT_SUSPEND_NS)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity; false when the limit passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// TMA gather of 4 rows (row coordinates r[0..3]) of a 2-D map whose box is
// one row of 64 elements; the rows land consecutively (4 x 128 B) at dst.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, const int (&r)[4], uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same with the A operand read from TMEM (M rows = lanes, K packed 2 per column).
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane; the wait is tied to
// the destination registers so no use is scheduled before it completes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout code 2), sm_100
// descriptor version 1.  lbo/sbo in bytes.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with fp32 accumulation.
__device__ __forceinline__ uint32_t idesc_f16(uint32_t bf16, uint32_t b_mn_major, int M, int N) {
  return (1u << 4) | (bf16 << 7) | (bf16 << 10) | (b_mn_major << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

template <typename Tout>
__device__ __forceinline__ void store_row(Tout* dst, const float* o, float inv);
template <>
__device__ __forceinline__ void store_row<float>(float* dst, const float* o, float inv) {
  float4* p = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                                  o[4 * i + 3] * inv);
}
template <>
__device__ __forceinline__ void store_row<__nv_bfloat16>(__nv_bfloat16* dst, const float* o, float inv) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 t = __floats2bfloat162_rn(o[8 * i + 2 * j] * inv, o[8 * i + 2 * j + 1] * inv);
      w[j] = *reinterpret_cast<uint32_t*>(&t);
    }
    p[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
template <>
__device__ __forceinline__ void store_row<__half>(__half* dst, const float* o, float inv) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 t = __floats2half2_rn(o[8 * i + 2 * j] * inv, o[8 * i + 2 * j + 1] * inv);
      w[j] = *reinterpret_cast<uint32_t*>(&t);
    }
    p[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One unit of work as every thread of the CTA sees it (all fields uniform).
struct Unit {
  int u, b, h, s0, n, q0, rows_q, nchunks;
};

// First unit at index >= u (stride `step`) whose query tile holds rows; a
// unit with an inconsistent length records an error and is skipped.
__device__ __forceinline__ Unit next_unit(int u, int step, int units, int BH, const AttendArgs& a, bool record) {
  Unit x;
  for (; u < units; u += step) {
    const int qt = u / BH;
    const int bh = u - qt * BH;
    const int h = bh % a.H;
    const int b = bh / a.H;
    const int s0 = __ldg(a.cu_seqlens + b);
    const int n = __ldg(a.cu_seqlens + b + 1) - s0;
    if (n < 0 || n > a.max_seqlen) {
      if (qt == 0 && h == 0 && record)
        record_error(a.err, n < 0 ? RRA_DEVERR_SEQ_NEGATIVE : RRA_DEVERR_SEQ_TOO_LONG);
      continue;
    }
    const int q0 = qt * BM;
    if (q0 >= n) continue;
    x.u = u;
    x.b = b;
    x.h = h;
    x.s0 = s0;
    x.n = n;
    x.q0 = q0;
    x.rows_q = min(BM, n - q0);
    x.nchunks = (n + BN - 1) / BN;
    return x;
  }
  x.u = units;
  return x;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(static_cast<unsigned short>(v)) : "memory");
}
__device__ __forceinline__ int ld_shared_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return static_cast<int>(v);
}

// Fused pipeline, called by the 32 lanes of the producer warp: the next unit
// at index >= u (stride `step`) whose query tile holds rows.  For every
// candidate the warp scans its image's keep row with ballots: the kept
// positions go, in order, to the int16 list at shared address `pos`; on the
// (image, head)'s first query tile the output rows of pruned positions are
// set to +0 (so every output row is written exactly once, images with no
// kept token included).
// Output rows (b, j, h) of pruned positions j -> +0 (producer warp, 32 lanes).
template <typename Tout>
__device__ __forceinline__ void zero_pruned_rows(const AttendArgs& a, int b, int h, int lane) {
  constexpr int OUT_VECS = HD * static_cast<int>(sizeof(Tout)) / 16;
  const uint8_t* krow = a.keep + static_cast<size_t>(b) * a.N;
  for (int j = lane; j < a.N; j += 32) {
    if (__ldg(krow + j) == 0) {
      uint4* row =
          reinterpret_cast<uint4*>(static_cast<Tout*>(a.o) + ((static_cast<size_t>(b) * a.N + j) * a.H + h) * HD);
#pragma unroll
      for (int v = 0; v < OUT_VECS; ++v) row[v] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Fused pipeline, called by the 32 lanes of the producer warp: the next unit
// at index >= u (stride `step`) whose query tile holds rows.  For every
// candidate the warp scans its image's keep row with ballots; the kept
// positions go, in order, to the int16 list at shared address `pos`.  A
// candidate skipped for having no rows in its tile zeroes its (image, head)'s
// pruned output rows here if it is the first query tile; the producer does
// the same for a returned first-tile unit once its loads are in flight, so
// every output row is written exactly once (images with no kept token too).
template <typename Tout>
__device__ Unit next_unit_fused(int u, int step, int units, int BH, const AttendArgs& a, int lane, uint32_t pos) {
  Unit x;
  const unsigned lt = (1u << lane) - 1u;
  for (; u < units; u += step) {
    const int qt = u / BH;
    const int bh = u - qt * BH;
    const int h = bh % a.H;
    const int b = bh / a.H;
    const uint8_t* krow = a.keep + static_cast<size_t>(b) * a.N;
    int cnt = 0;
    for (int j0 = 0; j0 < a.N; j0 += 8 * 32) {
      bool flag[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int j = j0 + r * 32 + lane;
        flag[r] = (j < a.N) && (__ldg(krow + j) != 0);
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int j = j0 + r * 32 + lane;
        const unsigned m = __ballot_sync(0xffffffffu, flag[r]);
        if (flag[r]) st_shared_u16(pos + 2u * static_cast<uint32_t>(cnt + __popc(m & lt)), static_cast<uint32_t>(j));
        cnt += __popc(m);
      }
    }
    const int q0 = qt * BM;
    if (q0 >= cnt) {
      if (qt == 0) zero_pruned_rows<Tout>(a, b, h, lane);
      continue;
    }
    x.u = u;
    x.b = b;
    x.h = h;
    x.s0 = 0;
    x.n = cnt;
    x.q0 = q0;
    x.rows_q = min(BM, cnt - q0);
    x.nchunks = (cnt + BN - 1) / BN;
    __syncwarp();
    return x;
  }
  x.u = units;
  return x;
}

// bf16 hi/lo split of two weights: hi = p truncated to bf16 (upper 16 bits,
// exact), lo = p - hi (exact in fp32) rounded to bf16; hi + lo carries p to
// 2^-16 relative.  Packed low half = first element (K order).
__device__ __forceinline__ void split2_bf16_trunc(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
  hi = __byte_perm(b0, b1, 0x7632);
  const float r0 = p0 - __uint_as_float(b0 & 0xFFFF0000u);
  const float r1 = p1 - __uint_as_float(b1 & 0xFFFF0000u);
  __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

// Exponentials of one S row chunk against reference mref, written back over
// S in TMEM as P hi/lo pairs (each 16-column piece of S becomes 8 hi + 8 lo
// columns in place); returns the chunk's row sum.  With ref_first the
// reference is replaced by this row's first score (so that weight is exactly
// 1: a one-token image returns V bit for bit) and written back to mref.
template <bool BF16>
__device__ __forceinline__ float chunk_weights(uint32_t tS_row, int nk16, int n_c, bool full, float c2, float& mref,
                                               bool ref_first) {
  float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int g = 0; g < BN / 16; ++g) {
    if (g * 16 < nk16) {
      float t[16];
      tmem_ld16(tS_row + g * 16, t);
      if (g == 0 && ref_first) mref = t[0] * c2;
      uint32_t hi[8], lo[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = g * 16 + 2 * i;
        float p0 = fast_exp2(fmaf(t[2 * i], c2, -mref));
        float p1 = fast_exp2(fmaf(t[2 * i + 1], c2, -mref));
        if (!full) {
          p0 = (j < n_c) ? p0 : 0.f;
          p1 = (j + 1 < n_c) ? p1 : 0.f;
        }
        l4[(2 * i) & 3] += p0;
        l4[(2 * i + 1) & 3] += p1;
        if constexpr (BF16) split2_bf16_trunc(p0, p1, hi[i], lo[i]);
        else split2<false>(p0, p1, hi[i], lo[i]);
      }
      tmem_st8(tS_row + g * 16, hi);
      tmem_st8(tS_row + g * 16 + 8, lo);
    }
  }
  return (l4[0] + l4[1]) + (l4[2] + l4[3]);
}

// Max of scale*S over the chunk's valid columns.
__device__ __forceinline__ float chunk_max(uint32_t tS_row, int nk16, int n_c, bool full, float c2) {
  float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int g = 0; g < BN / 16; ++g) {
    if (g * 16 < nk16) {
      float t[16];
      tmem_ld16(tS_row + g * 16, t);
      if (full) {
#pragma unroll
        for (int i = 0; i < 16; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], t[i] * c2);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (g * 16 + i < n_c) mx4[i & 3] = fmaxf(mx4[i & 3], t[i] * c2);
      }
    }
  }
  return fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
}

// O row (TMEM) *= alpha.
__device__ __forceinline__ void rescale_o(uint32_t tO_row, float alpha) {
#pragma unroll
  for (int g = 0; g < HD / 16; ++g) {
    float oc[16];
    tmem_ld16(tO_row + g * 16, oc);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(oc[i] * alpha);
    tmem_st8(tO_row + g * 16, w);
    tmem_st8(tO_row + g * 16 + 8, w + 8);
  }
}

// Consumer-only barrier (named barrier 1, the 128 consumer threads) that
// also ORs a predicate across them.
__device__ __forceinline__ bool consumer_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.or.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_volatile_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
// Bounded wait that also gives up as soon as the CTA's abort flag is set.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, uint32_t abort_flag) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (ld_shared_volatile_u32(abort_flag) != 0u) return false;
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) return false;
  }
  return true;
}

template <typename Tin, typename Tout, bool SCATTER, int MODE>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const AttendArgs a, int qtiles, int units,
                     int pos_stride) {
  constexpr bool BF = IsBf16<Tin>::value == 1;
  constexpr bool GATHER = MODE != MODE_PACKED;
  constexpr bool FUSED = MODE == MODE_FUSED;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + OFF_Q;
  auto sK = [&](int i) { return base + OFF_K + i * KV_BYTES; };
  auto sV = [&](int i) { return base + OFF_V + i * KV_BYTES; };
  auto bar_full = [&](int i) { return base + OFF_BAR + i * 8; };
  auto bar_empty = [&](int i) { return base + OFF_BAR + 16 + i * 8; };
  const uint32_t bar_qempty = base + OFF_BAR + 32, bar_mma = base + OFF_BAR + 40;
  const uint32_t slot = base + OFF_BAR + 48, abort_flag = base + OFF_BAR + 52;
  auto desc_addr = [&](int i) { return base + OFF_DESC + i * DESC_BYTES; };
  auto pos_addr = [&](int slot) { return base + OFF_POS + slot * pos_stride; };
  const volatile uint32_t* slot_ptr = reinterpret_cast<const volatile uint32_t*>(gbase + OFF_BAR + 48);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    tmem_alloc(slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    mbar_init(bar_qempty, 1);
    mbar_init(bar_mma, 1);
    st_shared_u32(abort_flag, 0u);
    st_shared_u32(base + OFF_BAR + 56, 0u);
    st_shared_u32(base + OFF_BAR + 60, 0u);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot_ptr;
  const int BH = a.B * a.H;
  const int step = gridDim.x;
  (void)qtiles;
  bool bad = false;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // Walks this CTA's items (unit, key chunk) in order.  For each: waits
    // until its stage (and, on a unit's first chunk, the Q buffer) is free,
    // publishes the item's descriptor, and issues the TMA loads that
    // complete the stage's full barrier.  Ends with a sentinel descriptor.
    uint32_t j = 0, uidx = 0;
    Unit U;
    if constexpr (FUSED) U = next_unit_fused<Tout>(blockIdx.x, step, units, BH, a, lane, pos_addr(0));
    else U = next_unit(blockIdx.x, step, units, BH, a, lane == 0);
    bool done = false;
    while (!done && !bad) {
      const int nch = (U.u < units) ? U.nchunks : 1;
      for (int c = 0; c < nch && !bad; ++c) {
        const int st = j & 1;
        if (j >= STAGES) bad |= !mbar_wait_or_abort(bar_empty(st), ((j >> 1) - 1) & 1, abort_flag);
        if (U.u < units && c == 0 && uidx >= 1)
          bad |= !mbar_wait_or_abort(bar_qempty, (uidx - 1) & 1, abort_flag);
        bad = __any_sync(0xffffffffu, bad);
        if (bad) break;
        if (U.u >= units) {
          // Sentinel: no more items.
          if (lane == 0) {
            st_shared_u32(desc_addr(st), static_cast<uint32_t>(units));
            mbar_arrive(bar_full(st));
          }
          done = true;
          break;
        }
        const int k0 = c * BN;
        const int n_c = min(BN, U.n - k0);
        if (lane == 0) {
          const uint32_t d = desc_addr(st);
          st_shared_u32(d + 0, static_cast<uint32_t>(U.u));
          st_shared_u32(d + 4, static_cast<uint32_t>(U.h));
          st_shared_u32(d + 8, static_cast<uint32_t>(U.s0));
          st_shared_u32(d + 12, static_cast<uint32_t>(U.n));
          st_shared_u32(d + 16, static_cast<uint32_t>(U.q0));
          st_shared_u32(d + 20, static_cast<uint32_t>(U.rows_q));
          st_shared_u32(d + 24, static_cast<uint32_t>(U.nchunks));
          st_shared_u32(d + 28, static_cast<uint32_t>(c));
          st_shared_u32(d + 32, static_cast<uint32_t>(U.b));
          st_shared_u32(d + 36, static_cast<uint32_t>(uidx % POS_SLOTS));
        }
        if constexpr (GATHER) {
          const int kgroups = ((n_c + 15) & ~15) / 4;
          const int qgroups = (c == 0) ? (U.rows_q + 3) / 4 : 0;
          if (lane == 0) mbar_expect_tx(bar_full(st), static_cast<uint32_t>((2 * kgroups + qgroups) * 512));
          __syncwarp();
          if (lane < qgroups) {
            int rows[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int t = min(U.q0 + 4 * lane + i, U.q0 + U.rows_q - 1);
              if constexpr (FUSED)
                rows[i] = (U.b * a.N + ld_shared_u16(pos_addr(uidx % POS_SLOTS) + 2 * t)) * a.H + U.h;
              else
                rows[i] = __ldg(a.src_idx + U.s0 + t) * a.H + U.h;
            }
            tma_gather4(sQ + lane * 512, &tmap_q, rows, bar_full(st));
          }
          const int g = lane & 15;
          if (g < kgroups) {
            int rows[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int t = min(k0 + 4 * g + i, k0 + n_c - 1);
              if constexpr (FUSED)
                rows[i] = (U.b * a.N + ld_shared_u16(pos_addr(uidx % POS_SLOTS) + 2 * t)) * a.H + U.h;
              else
                rows[i] = __ldg(a.src_idx + U.s0 + t) * a.H + U.h;
            }
            if (lane < 16) tma_gather4(sK(st) + g * 512, &tmap_k, rows, bar_full(st));
            else tma_gather4(sV(st) + g * 512, &tmap_v, rows, bar_full(st));
          }
        } else if (lane == 0) {
          const int kboxes = (n_c + BOX - 1) / BOX;
          const int qboxes = (c == 0) ? (U.rows_q + BOX - 1) / BOX : 0;
          mbar_expect_tx(bar_full(st), static_cast<uint32_t>((2 * kboxes + qboxes) * BOX * 128));
          for (int jj = 0; jj < qboxes; ++jj)
            tma_load_3d(sQ + jj * BOX * 128, &tmap_q, 0, U.h, U.s0 + U.q0 + jj * BOX, bar_full(st));
          for (int jj = 0; jj < kboxes; ++jj) {
            tma_load_3d(sK(st) + jj * BOX * 128, &tmap_k, 0, U.h, U.s0 + k0 + jj * BOX, bar_full(st));
            tma_load_3d(sV(st) + jj * BOX * 128, &tmap_v, 0, U.h, U.s0 + k0 + jj * BOX, bar_full(st));
          }
        }
        __syncwarp();
        if constexpr (FUSED) {
          // The unit's first loads are in flight: now zero its (image,
          // head)'s pruned output rows if this is the first query tile.
          if (c == 0 && U.q0 == 0) zero_pruned_rows<Tout>(a, U.b, U.h, lane);
        }
        ++j;
      }
      if (done || bad) break;
      ++uidx;
      if constexpr (FUSED) U = next_unit_fused<Tout>(U.u + step, step, units, BH, a, lane, pos_addr(uidx % POS_SLOTS));
      else U = next_unit(U.u + step, step, units, BH, a, lane == 0);
    }
    if (!bad) {
      // Tail: wait for the consumers' last stage and Q releases, so that no
      // asynchronous arrive lands after the CTA has gone.
      if (j >= 1) bad |= !mbar_wait_or_abort(bar_empty((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag);
      if (uidx >= 1) bad |= !mbar_wait_or_abort(bar_qempty, (uidx - 1) & 1, abort_flag);
      bad = __any_sync(0xffffffffu, bad);
    }
    if (bad) {
      if (lane == 0) {
        st_shared_u32(abort_flag, 1u);
        record_error(a.err, RRA_DEVERR_WAIT_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem, tO = tmem + 64;
    const uint32_t tS_row = tS + lane_off, tO_row = tO + lane_off;
    const uint32_t idesc_pv = idesc_f16(BF ? 1u : 0u, 1, BM, HD);
    const float c2 = a.scale_log2;
    uint32_t ph_mma = 0;
    float m_run = 0.f, l_run = 0.f;   // this row's reference max (log2 units) and sum
    for (uint32_t j = 0;; ++j) {
      const int st = j & 1;
      bad |= !mbar_wait_or_abort(bar_full(st), (j >> 1) & 1, abort_flag);
      if (consumer_sync_or(bad)) { bad = true; break; }
      const uint32_t d = desc_addr(st);
      const int u = static_cast<int>(ld_shared_u32(d + 0));
      if (u >= units) break;   // sentinel
      const int h = static_cast<int>(ld_shared_u32(d + 4));
      const int s0 = static_cast<int>(ld_shared_u32(d + 8));
      const int n = static_cast<int>(ld_shared_u32(d + 12));
      const int q0 = static_cast<int>(ld_shared_u32(d + 16));
      const int rows_q = static_cast<int>(ld_shared_u32(d + 20));
      const int nchunks = static_cast<int>(ld_shared_u32(d + 24));
      const int c = static_cast<int>(ld_shared_u32(d + 28));
      const int b = static_cast<int>(ld_shared_u32(d + 32));
      const int pslot = static_cast<int>(ld_shared_u32(d + 36));
      const int k0 = c * BN;
      const int n_c = min(BN, n - k0);
      const int nk16 = (n_c + 15) & ~15;
      const bool full = (n_c == BN);
      const bool rows_here = warp * 32 < rows_q;   // warp-uniform
      const bool last = (c == nchunks - 1);

      // S = Q K^T -> TMEM columns [0, nk16).  Packed inputs: warp 0 first
      // zeroes the V rows [n_c, nk16) that enter the MMA with p = 0 (the
      // gathered path repeats a finite row there instead).
      if (warp == 0) {
        if constexpr (!GATHER) {
          const int zvec = (nk16 - n_c) * 8;
          for (int zi = lane; zi < zvec; zi += 32)
            st_shared_v4(sV(st) + (n_c + (zi >> 3)) * 128 + (zi & 7) * 16, 0u, 0u, 0u, 0u);
          fence_proxy_async();
          __syncwarp();
        }
        if (tid == 0) {
          tc_fence_after();
          const uint32_t idesc_s = idesc_f16(BF ? 1u : 0u, 0, BM, nk16);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_f16(tS, sdesc(sQ + kk * 32, 16, 1024), sdesc(sK(st) + kk * 32, 16, 1024), idesc_s,
                     kk > 0 ? 1u : 0u);
          umma_commit(bar_mma);
        }
      }
      bad |= !mbar_wait_or_abort(bar_mma, ph_mma, abort_flag);
      if (!bad) ph_mma ^= 1;
      bad = __any_sync(0xffffffffu, bad);   // warp-uniform before warp-collective TMEM access
      tc_fence_after();

      // Softmax on this thread's row (TMEM lane).  Exponentials are taken
      // against a per-row reference m_run (log2 units) and O accumulates in
      // TMEM across chunks.  bf16: one pass, the reference being the row's
      // first score on the first chunk and the running reference after, P
      // written over S at once; a row whose chunk sum exceeds 2^32 flags a
      // redo, and then the consumers recompute S and this chunk (exact max
      // and O rescale for the flagged rows).  fp16 (narrower range for P):
      // max pass first, rescale when the max grows by > 8.
      const float l_before = l_run, m_before = m_run;
      // Redo flag of this item: two words used alternately, set to j + 1,
      // so a stale value from two items back never reads as set.
      const uint32_t flag = base + OFF_BAR + 56 + (j & 1) * 4;
      bool redo_row = false;
      if (rows_here && !bad) {
        if constexpr (BF) {
          l_run += chunk_weights<true>(tS_row, nk16, n_c, full, c2, m_run, c == 0);
          redo_row = (tid < rows_q) && !(l_run - l_before <= 0x1p32f);
          if (__any_sync(0xffffffffu, redo_row) && lane == 0) st_shared_u32(flag, j + 1u);
        } else {
          const float mx = chunk_max(tS_row, nk16, n_c, full, c2);
          if (c == 0) {
            m_run = mx;
          } else if (__any_sync(0xffffffffu, mx > m_run + 8.f)) {
            const float m_new = fmaxf(m_run, mx);
            const float alpha = fast_exp2(m_run - m_new);
            l_run *= alpha;
            rescale_o(tO_row, alpha);
            m_run = m_new;
          }
          l_run += chunk_weights<false>(tS_row, nk16, n_c, full, c2, m_run, false);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      if (consumer_sync_or(bad)) { bad = true; break; }
      if (BF && ld_shared_u32(flag) == j + 1u) {
        // Rare: recompute S, then every warp rewrites its P; flagged warps
        // switch to the exact max (rescaling O for later chunks).
        if (tid == 0) {
          tc_fence_after();
          const uint32_t idesc_s = idesc_f16(BF ? 1u : 0u, 0, BM, nk16);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_f16(tS, sdesc(sQ + kk * 32, 16, 1024), sdesc(sK(st) + kk * 32, 16, 1024), idesc_s,
                     kk > 0 ? 1u : 0u);
          umma_commit(bar_mma);
        }
        bad |= !mbar_wait_or_abort(bar_mma, ph_mma, abort_flag);
        if (!bad) ph_mma ^= 1;
        bad = __any_sync(0xffffffffu, bad);
        tc_fence_after();
        if (rows_here && !bad) {
          l_run = l_before;
          m_run = m_before;
          if (__any_sync(0xffffffffu, redo_row)) {
            const float mx = chunk_max(tS_row, nk16, n_c, full, c2);
            const float m_new = (c == 0) ? mx : fmaxf(m_before, mx);
            if (c > 0) {
              const float alpha = fast_exp2(m_before - m_new);
              l_run *= alpha;
              rescale_o(tO_row, alpha);
            }
            m_run = m_new;
            l_run += chunk_weights<true>(tS_row, nk16, n_c, full, c2, m_run, false);
          } else {
            l_run += chunk_weights<true>(tS_row, nk16, n_c, full, c2, m_run, c == 0);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        if (consumer_sync_or(bad)) { bad = true; break; }
      }

      // O += P_hi V + P_lo V in TMEM columns [64, 128) (fresh on a unit's
      // first chunk).  Its completion frees this K/V stage for the producer
      // and, on the unit's last chunk, the Q buffer.
      if (tid == 0) {
        tc_fence_after();
        const int ksteps = nk16 / 16;
        for (int kk = 0; kk < ksteps; ++kk)
          umma_f16_tmem_a(tO, tS + kk * 16, sdesc(sV(st) + kk * 2048, KV_BYTES, 1024), idesc_pv,
                          (kk > 0 || c > 0) ? 1u : 0u);
        for (int kk = 0; kk < ksteps; ++kk)
          umma_f16_tmem_a(tO, tS + kk * 16 + 8, sdesc(sV(st) + kk * 2048, KV_BYTES, 1024), idesc_pv, 1u);
        umma_commit(bar_empty(st));
        if (last) umma_commit(bar_qempty);
        umma_commit(bar_mma);
      }
      bad |= !mbar_wait_or_abort(bar_mma, ph_mma, abort_flag);
      if (!bad) ph_mma ^= 1;
      bad = __any_sync(0xffffffffu, bad);
      tc_fence_after();

      if (last && rows_here && !bad) {
        // Epilogue: this thread's row, normalised, to the packed or padded output.
        float o_acc[HD];
#pragma unroll
        for (int g = 0; g < HD / 16; ++g) tmem_ld16(tO_row + g * 16, o_acc + g * 16);
        const int i = q0 + tid;
        if (i < n) {
          long long dst_row = static_cast<long long>(s0) + i;
          bool ok = true;
          if constexpr (FUSED) {
            dst_row = static_cast<long long>(b) * a.N + ld_shared_u16(pos_addr(pslot) + 2 * i);
          } else if constexpr (SCATTER) {
            dst_row = __ldg(a.src_idx + dst_row);
            if (dst_row < 0 || dst_row >= static_cast<long long>(a.B) * a.N) {
              record_error(a.err, RRA_DEVERR_INDEX_RANGE);
              ok = false;
            }
          }
          if (ok) {
            Tout* out = static_cast<Tout*>(a.o) + (static_cast<size_t>(dst_row) * a.H + h) * HD;
            store_row<Tout>(out, o_acc, 1.f / l_run);
          }
        }
      }
      if (last) {
        m_run = 0.f;
        l_run = 0.f;
      }
      // No barrier here: the next S product overwrites S/P only after thread
      // 0 has seen this P.V product complete, and the next unit's first P.V
      // (which overwrites O) waits behind the next P-ready barrier.
    }
    if (bad && tid == 0) {
      st_shared_u32(abort_flag, 1u);
      record_error(a.err, RRA_DEVERR_WAIT_TIMEOUT);
    }
  }

  // Teardown.  After an abort, copies or MMAs still in flight get a bounded
  // grace period (~1 ms) to land before the TMEM is released and the CTA exits.
  if (ld_shared_volatile_u32(abort_flag) != 0u && tid == 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < 2000000LL) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 3-D map over a packed [rows, H, 64] tensor: box = 32 rows of one head.
cudaError_t make_map(CUtensorMap* map, const void* ptr, int H, long long rows, bool bf16) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(HD * 2), static_cast<cuuint64_t>(H) * HD * 2};
  cuuint32_t box[3] = {HD, 1, BOX};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                        const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

constexpr int kMaxDev = 64;

// 2-D map over a padded [B*N*H, 64] tensor with a one-row box, for gather4.
cudaError_t make_gather_map(CUtensorMap* map, const void* ptr, long long rows, bool bf16) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(HD * 2)};
  cuuint32_t box[2] = {HD, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                        const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename Tin, typename Tout, bool SCATTER, int MODE>
cudaError_t launch_tc_typed(const AttendArgs& a, int num_sms, cudaStream_t stream) {
  // Largest dynamic shared memory any launch of this instantiation asks for
  // (position lists for N <= 1024 in the fused mode).
  constexpr uint32_t kMaxSmem = SMEM_ALLOC + (MODE == MODE_FUSED ? POS_SLOTS * 2048u : 0u);
  static bool attr_set[kMaxDev] = {};
  static std::mutex m;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(m);
    if (!attr_set[dev]) {
      e = cudaFuncSetAttribute(attend_tc_kernel<Tin, Tout, SCATTER, MODE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxSmem));
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  const bool bf16 = IsBf16<Tin>::value == 1;
  CUtensorMap mq, mk, mv;
  if constexpr (MODE != MODE_PACKED) {
    const long long rows = static_cast<long long>(a.B) * a.N * a.H;
    if ((e = make_gather_map(&mq, a.qp, rows, bf16)) != cudaSuccess) return e;
    if ((e = make_gather_map(&mk, a.kp, rows, bf16)) != cudaSuccess) return e;
    if ((e = make_gather_map(&mv, a.vp, rows, bf16)) != cudaSuccess) return e;
  } else {
    const long long rows = static_cast<long long>(a.B) * a.max_seqlen;
    if ((e = make_map(&mq, a.qp, a.H, rows, bf16)) != cudaSuccess) return e;
    if ((e = make_map(&mk, a.kp, a.H, rows, bf16)) != cudaSuccess) return e;
    if ((e = make_map(&mv, a.vp, a.H, rows, bf16)) != cudaSuccess) return e;
  }
  const int pos_stride = (MODE == MODE_FUSED) ? ((2 * a.N + 15) & ~15) : 0;
  const uint32_t smem = SMEM_ALLOC + static_cast<uint32_t>(POS_SLOTS * pos_stride);
  const int qtiles = (a.max_seqlen + BM - 1) / BM;
  const long long units = static_cast<long long>(a.B) * a.H * qtiles;
  const long long cap = static_cast<long long>(CTAS_PER_SM) * (num_sms > 0 ? num_sms : 152);
  const int grid = static_cast<int>(units < cap ? units : cap);
  attend_tc_kernel<Tin, Tout, SCATTER, MODE><<<grid, THREADS, smem, stream>>>(mq, mk, mv, a, qtiles,
                                                                             static_cast<int>(units), pos_stride);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_tc_out(const AttendArgs& a, int mode, int num_sms, cudaStream_t stream) {
  if (mode == MODE_FUSED) return launch_tc_typed<Tin, Tout, true, MODE_FUSED>(a, num_sms, stream);
  if (mode == MODE_GATHER) return launch_tc_typed<Tin, Tout, true, MODE_GATHER>(a, num_sms, stream);
  if (a.src_idx != nullptr) return launch_tc_typed<Tin, Tout, true, MODE_PACKED>(a, num_sms, stream);
  return launch_tc_typed<Tin, Tout, false, MODE_PACKED>(a, num_sms, stream);
}

template <typename Tin>
cudaError_t launch_tc_in(const AttendArgs& a, rra_dtype out, int mode, int num_sms, cudaStream_t stream) {
  if (out == RRA_BF16) return launch_tc_out<Tin, __nv_bfloat16>(a, mode, num_sms, stream);
  if (out == RRA_F16) return launch_tc_out<Tin, __half>(a, mode, num_sms, stream);
  return launch_tc_out<Tin, float>(a, mode, num_sms, stream);
}

}  // namespace

bool attend_tc_available() { return encode_fn(); }

cudaError_t launch_attend_tc(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms, cudaStream_t stream) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (static_cast<long long>(a.B) * a.max_seqlen >= (1LL << 31)) return cudaErrorInvalidValue;
  if (in == RRA_BF16) return launch_tc_in<__nv_bfloat16>(a, out, MODE_PACKED, num_sms, stream);
  return launch_tc_in<__half>(a, out, MODE_PACKED, num_sms, stream);
}

cudaError_t launch_attend_tc_gather(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                    cudaStream_t stream) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (a.src_idx == nullptr) return cudaErrorInvalidValue;
  if (in == RRA_BF16) return launch_tc_in<__nv_bfloat16>(a, out, MODE_GATHER, num_sms, stream);
  return launch_tc_in<__half>(a, out, MODE_GATHER, num_sms, stream);
}

cudaError_t launch_attend_tc_fused(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                   cudaStream_t stream) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (a.keep == nullptr || a.N > 1024) return cudaErrorInvalidValue;
  if (in == RRA_BF16) return launch_tc_in<__nv_bfloat16>(a, out, MODE_FUSED, num_sms, stream);
  return launch_tc_in<__half>(a, out, MODE_FUSED, num_sms, stream);
}

}  // namespace rra

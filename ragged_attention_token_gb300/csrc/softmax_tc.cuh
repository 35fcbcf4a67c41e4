// Softmax and output building blocks shared by the tcgen05 attention
// kernels: base-2 exponentials, the per-row extreme of a 32-column group of
// S, the weights written back over S as two 16-bit parts (hi + lo), the
// rescale of O and of written weights when a row's reference moves, the
// softmax of one 64-key chunk for one query row, and the output stores.
// Inline device code only (each kernel file gets its own copy).
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace rra {
namespace {

constexpr int HD = 64;   // head dim

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

template <typename Tout>
__device__ __forceinline__ void store16(Tout* dst, const float* o, float inv);
template <>
__device__ __forceinline__ void store16<float>(float* dst, const float* o, float inv) {
  float4* p = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    p[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
}
template <typename T2>
__device__ __forceinline__ uint32_t pack2(float x, float y);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat162>(float x, float y) {
  __nv_bfloat162 t = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&t);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half2>(float x, float y) {
  __half2 t = __floats2half2_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&t);
}
template <typename T2>
__device__ __forceinline__ void store16_half(void* dst, const float* o, float inv) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    p[i] = make_uint4(pack2<T2>(o[8 * i] * inv, o[8 * i + 1] * inv), pack2<T2>(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                      pack2<T2>(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                      pack2<T2>(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
}
// The packed-pair type of a 16-bit output type.
template <typename T> struct Tout2Of;
template <> struct Tout2Of<__nv_bfloat16> { using type = __nv_bfloat162; };
template <> struct Tout2Of<__half> { using type = __half2; };
template <> struct Tout2Of<float> { using type = __nv_bfloat162; };   // unused
template <typename T> using Tout2 = typename Tout2Of<T>::type;

template <>
__device__ __forceinline__ void store16<__nv_bfloat16>(__nv_bfloat16* dst, const float* o, float inv) {
  store16_half<__nv_bfloat162>(dst, o, inv);
}
template <>
__device__ __forceinline__ void store16<__half>(__half* dst, const float* o, float inv) {
  store16_half<__half2>(dst, o, inv);
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(static_cast<unsigned short>(v)) : "memory");
}
__device__ __forceinline__ int ld_shared_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return static_cast<int>(v);
}

// Output rows (b, j, h) of image b's pruned positions j for this head -> +0,
// with plain stores (producer warp, 32 lanes).  The mask bytes of 256
// positions are loaded together before any store.  Used when the grid has at
// most one unit per SM: there the plain stores finish sooner than bulk copies.
template <typename Tout>
__device__ __forceinline__ void zero_pruned_rows(const AttendArgs& a, int b, int h, int lane) {
  constexpr int OUT_VECS = HD * static_cast<int>(sizeof(Tout)) / 16;
  const uint8_t* krow = a.keep + static_cast<size_t>(b) * a.N;
  for (int j0 = 0; j0 < a.N; j0 += 8 * 32) {
    bool pruned[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int j = j0 + r * 32 + lane;
      pruned[r] = (j < a.N) && (__ldg(krow + j) == 0);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (pruned[r]) {
        const size_t j = static_cast<size_t>(j0 + r * 32 + lane);
        uint4* row = reinterpret_cast<uint4*>(static_cast<Tout*>(a.o) + ((static_cast<size_t>(b) * a.N + j) * a.H + h) * HD);
#pragma unroll
        for (int v = 0; v < OUT_VECS; ++v) row[v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

// Three-input max / min (one instruction each on sm_100 and later).
__device__ __forceinline__ float max3f(float x, float y, float z) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(x), "f"(y), "f"(z));
  return d;
}
__device__ __forceinline__ float min3f(float x, float y, float z) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(x), "f"(y), "f"(z));
  return d;
}

// Packed pairs of fp32 (sm_100 and later execute fma/add/sub on both halves
// of a 64-bit register pair in one instruction).
__device__ __forceinline__ uint64_t pack_f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack_f2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Weights of one 32-column group of a chunk row, p = 2^(c2*s - mref) (0 at
// columns >= nvalid when !full), written back over S in TMEM as hi/lo pairs
// (each 16-column piece of S becomes 8 hi + 8 lo columns in place); returns
// their sum.  Only the first 16 columns when cols == 16.
// bf16: hi = p truncated to bf16 (exact), lo = p - hi (exact in fp32)
// rounded to bf16; fp16: hi = p rounded to fp16, lo = p - hi rounded.
template <bool BF16>
__device__ __forceinline__ float weights32(uint32_t tS, const float (&t)[32], int cols, int nvalid, bool full,
                                          float c2, float mref) {
  const uint64_t c2x2 = pack_f2(c2, c2), nm2 = pack_f2(-mref, -mref);
  uint64_t acc[2] = {0ull, 0ull};   // packed partial sums (+0.0f pairs)
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    if (g == 0 || cols > 16) {
      uint32_t hi[8], lo[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int col = 16 * g + 2 * i;
        float x0, x1;
        unpack_f2(fma_f2(pack_f2(t[col], t[col + 1]), c2x2, nm2), x0, x1);
        float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
        if (!full) {
          p0 = (col < nvalid) ? p0 : 0.f;
          p1 = (col + 1 < nvalid) ? p1 : 0.f;
        }
        const uint64_t pp = pack_f2(p0, p1);
        acc[i & 1] = add_f2(acc[i & 1], pp);
        float r0, r1;
        if constexpr (BF16) {
          const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
          hi[i] = __byte_perm(b0, b1, 0x7632);
          unpack_f2(sub_f2(pp, pack_f2(__uint_as_float(b0 & 0xFFFF0000u), __uint_as_float(b1 & 0xFFFF0000u))), r0,
                    r1);
          __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
          lo[i] = *reinterpret_cast<uint32_t*>(&l);
        } else {
          const __half2 h = __floats2half2_rn(p0, p1);
          hi[i] = *reinterpret_cast<const uint32_t*>(&h);
          unpack_f2(sub_f2(pp, pack_f2(__low2float(h), __high2float(h))), r0, r1);
          const __half2 l = __floats2half2_rn(r0, r1);
          lo[i] = *reinterpret_cast<const uint32_t*>(&l);
        }
      }
      tmem_st8(tS + g * 16, hi);
      tmem_st8(tS + g * 16 + 8, lo);
    }
  }
  float s0, s1, s2, s3;
  unpack_f2(acc[0], s0, s1);
  unpack_f2(acc[1], s2, s3);
  return (s0 + s1) + (s2 + s3);
}

// Largest (LOW: smallest) raw score over the first nvalid columns of a
// 32-column group; the others are first replaced by -inf (LOW: +inf).
template <bool LOW>
__device__ __forceinline__ float group_extreme(float (&t)[32], int nvalid) {
  const float pad = LOW ? INFINITY : -INFINITY;
  if (nvalid < 32) {
#pragma unroll
    for (int i = 0; i < 32; ++i) t[i] = (i < nvalid) ? t[i] : pad;
  }
  float e[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float* s = t + 8 * k;
    if constexpr (LOW) e[k] = fminf(min3f(min3f(min3f(s[0], s[1], s[2]), s[3], s[4]), s[5], s[6]), s[7]);
    else e[k] = fmaxf(max3f(max3f(max3f(s[0], s[1], s[2]), s[3], s[4]), s[5], s[6]), s[7]);
  }
  return LOW ? fminf(min3f(e[0], e[1], e[2]), e[3]) : fmaxf(max3f(e[0], e[1], e[2]), e[3]);
}

// 32 (or 16, the rest set to 0) columns of this thread's S row.
__device__ __forceinline__ void load_group(uint32_t taddr, int cols, float (&t)[32]) {
  if (cols > 16) {
    tmem_ld32(taddr, t);
  } else {
    tmem_ld16(taddr, t);
#pragma unroll
    for (int i = 16; i < 32; ++i) t[i] = 0.f;
  }
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

// The 32 columns of P already written for the first key group (two pieces
// of 8 hi + 8 lo columns) times alpha, split again the same way.
template <bool BF16>
__device__ __forceinline__ void rescale_p32(uint32_t tS_row, float alpha) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    float raw[16];
    tmem_ld16(tS_row + g * 16, raw);
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t h = __float_as_uint(raw[i]), l = __float_as_uint(raw[8 + i]);
      float p0, p1;
      if constexpr (BF16) {
        p0 = (__uint_as_float(h << 16) + __uint_as_float(l << 16)) * alpha;
        p1 = (__uint_as_float(h & 0xFFFF0000u) + __uint_as_float(l & 0xFFFF0000u)) * alpha;
        const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
        hi[i] = __byte_perm(b0, b1, 0x7632);
        __nv_bfloat162 r = __floats2bfloat162_rn(p0 - __uint_as_float(b0 & 0xFFFF0000u),
                                                 p1 - __uint_as_float(b1 & 0xFFFF0000u));
        lo[i] = *reinterpret_cast<uint32_t*>(&r);
      } else {
        const __half2 hh = *reinterpret_cast<const __half2*>(&h), ll = *reinterpret_cast<const __half2*>(&l);
        p0 = (__low2float(hh) + __low2float(ll)) * alpha;
        p1 = (__high2float(hh) + __high2float(ll)) * alpha;
        const __half2 nh = __floats2half2_rn(p0, p1);
        const __half2 nl = __floats2half2_rn(p0 - __low2float(nh), p1 - __high2float(nh));
        hi[i] = *reinterpret_cast<const uint32_t*>(&nh);
        lo[i] = *reinterpret_cast<const uint32_t*>(&nl);
      }
    }
    tmem_st8(tS_row + g * 16, hi);
    tmem_st8(tS_row + g * 16 + 8, lo);
  }
}


// The raw scores of one group of a row (16 or 32 columns) to global memory,
// 16 bytes per store (dst 16-byte aligned).
__device__ __forceinline__ void stash_row(float* dst, const float (&t)[32], int cols) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < 4 || cols > 16) d4[i] = make_float4(t[4 * i], t[4 * i + 1], t[4 * i + 2], t[4 * i + 3]);
}

// Softmax of one 64-key chunk (nk16 columns of S, the first n_c valid) for
// this thread's query row, in two 32-column groups: each group's row max
// (from the registers it was loaded into), then its weights written over S.
// The reference m moves only when a group's max exceeds it by more than 8 in
// the log2 domain: O (the finished products of the earlier chunks) and l are
// rescaled, and so is the group of P already written.  So every weight stays
// below 2^8.  On a unit's first chunk (c == 0) m and l start from this chunk.
// `vote`: this thread's row is one of the tile's rows (only those may move
// the reference; lanes past the tile see whatever the Q buffer held).
// CLS: a thread given `stash` (not null) also stores its row's raw scores of
// the chunk's nk16 columns there.
template <bool BF, bool CLS = false>
__device__ __forceinline__ void softmax_chunk64(uint32_t tS_row, uint32_t tO_row, int nk16, int n_c, int c,
                                                bool vote, float c2, float& m_run, float& l_run,
                                                float* stash = nullptr) {
  const int cols_a = min(32, nk16), cols_b = nk16 - 32;
  const int va = min(32, n_c), vb = n_c - 32;
  float m = m_run;
  float t[32];
  load_group(tS_row, cols_a, t);
  if constexpr (CLS) {
    if (stash != nullptr) stash_row(stash, t, cols_a);
  }
  {
    const float e = (c2 >= 0.f ? group_extreme<false>(t, va) : group_extreme<true>(t, va)) * c2;
    if (c == 0) {
      m = e;
      l_run = 0.f;
    } else if (__any_sync(0xffffffffu, vote && e > m + 8.f)) {
      const float m_new = fmaxf(m, e);
      const float alpha = fast_exp2(m - m_new);
      l_run *= alpha;
      rescale_o(tO_row, alpha);
      m = m_new;
      load_group(tS_row, cols_a, t);   // not kept across the rescale
    }
    l_run += weights32<BF>(tS_row, t, cols_a, va, va >= 32, c2, m);
  }
  if (cols_b > 0) {
    load_group(tS_row + 32, cols_b, t);
    if constexpr (CLS) {
      if (stash != nullptr) stash_row(stash + 32, t, cols_b);
    }
    const float e = (c2 >= 0.f ? group_extreme<false>(t, vb) : group_extreme<true>(t, vb)) * c2;
    if (__any_sync(0xffffffffu, vote && e > m + 8.f)) {
      const float m_new = fmaxf(m, e);
      const float alpha = fast_exp2(m - m_new);
      l_run *= alpha;
      if (c > 0) rescale_o(tO_row, alpha);
      tmem_st_wait();
      rescale_p32<BF>(tS_row, alpha);
      m = m_new;
      load_group(tS_row + 32, cols_b, t);
    }
    l_run += weights32<BF>(tS_row + 32, t, cols_b, vb, vb >= 32, c2, m);
  }
  m_run = m;
  tmem_st_wait();
}

}  // namespace
}  // namespace rra

// Fused token packing: keep mask -> cu_seqlens, dst_idx, src_idx, and a
// 128-bit gather of the kept Q/K/V rows into the flat packed buffers.
//
// Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers",
// agents-report.net article, section "方法概覽" (method overview), bullet 1:
// index work on the GPU produces the per-image offsets and destination
// indices, then a vectorised copy gathers the surviving tokens.
//
// Design.  Packed order is batch order then token order, so the packed row
// of flat position g = b*N + j is simply the number of kept tokens at flat
// positions < g: the whole pack is one stream compaction over B*N tokens.
// Each CTA owns a contiguous token range [g0, g1).  It obtains the exclusive
// count at g0 by counting nonzero mask bytes in keep[0, g0) with 16-byte
// loads (the mask is small and L2-resident; the grid is capped at a few CTAs
// per SM so the redundant counting stays far below the copy traffic), then
// ranks its own tokens with warp ballots.  No CTA waits on another, so there
// is no inter-CTA spin and no second launch.  cu_seqlens[b] is the exclusive
// count at g = b*N.  Row copies are 16-byte loads/stores, consecutive
// threads on consecutive vectors of a row.
#include "common.cuh"

namespace rra {

constexpr int PACK_THREADS = 256;
constexpr int PACK_WARPS = PACK_THREADS / 32;

__device__ __forceinline__ int nonzero_bytes(uint32_t x) {
  // bit 7 of each byte of t is set iff that byte of x is nonzero
  uint32_t t = ((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x;
  return __popc(t & 0x80808080u);
}

__device__ __forceinline__ int nonzero_bytes(uint4 w) {
  return nonzero_bytes(w.x) + nonzero_bytes(w.y) + nonzero_bytes(w.z) + nonzero_bytes(w.w);
}

// Number of nonzero bytes in keep[0, n), summed over the block (all threads
// receive the total).  `red` is PACK_WARPS ints of shared memory.
__device__ int block_count_prefix(const uint8_t* __restrict__ keep, long long n, int* red) {
  int c = 0;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(keep);
  long long head = static_cast<long long>((16 - (addr & 15)) & 15);
  if (head > n) head = n;
  for (long long i = threadIdx.x; i < head; i += PACK_THREADS) c += keep[i] != 0;
  const uint4* vec = reinterpret_cast<const uint4*>(keep + head);
  const long long nv = (n - head) >> 4;
  long long i = threadIdx.x;
  for (; i + 3 * PACK_THREADS < nv; i += 4 * PACK_THREADS) {
    uint4 w0 = __ldg(vec + i);
    uint4 w1 = __ldg(vec + i + PACK_THREADS);
    uint4 w2 = __ldg(vec + i + 2 * PACK_THREADS);
    uint4 w3 = __ldg(vec + i + 3 * PACK_THREADS);
    c += nonzero_bytes(w0) + nonzero_bytes(w1) + nonzero_bytes(w2) + nonzero_bytes(w3);
  }
  for (; i < nv; i += PACK_THREADS) c += nonzero_bytes(__ldg(vec + i));
  for (long long t = head + nv * 16 + threadIdx.x; t < n; t += PACK_THREADS) c += keep[t] != 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = c;
  __syncthreads();
  int total = 0;
#pragma unroll
  for (int w = 0; w < PACK_WARPS; ++w) total += red[w];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(PACK_THREADS) pack_kernel(const PackArgs a) {
  __shared__ int s_red[PACK_WARPS];
  __shared__ int s_kept_cnt[PACK_WARPS];
  __shared__ int s_pruned_cnt[PACK_WARPS];
  __shared__ long long s_kept_src[PACK_THREADS];   // source row of the copy, -1: none
  __shared__ int s_kept_dst[PACK_THREADS];
  __shared__ int s_pruned_g[PACK_THREADS];

  const long long total = static_cast<long long>(a.B) * a.N;
  const long long g0 = static_cast<long long>(blockIdx.x) * a.tok_per_cta;
  if (g0 >= total) return;
  const long long g1 = min(g0 + a.tok_per_cta, total);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;

  int running = block_count_prefix(a.keep, g0, s_red);

  for (long long r0 = g0; r0 < g1; r0 += PACK_THREADS) {
    const long long g = r0 + threadIdx.x;
    const bool valid = g < g1;
    const bool kept = valid && a.keep[g] != 0;
    const bool pruned = valid && !kept;
    const unsigned kb = __ballot_sync(0xffffffffu, kept);
    const unsigned pb = __ballot_sync(0xffffffffu, pruned);
    if (lane == 0) {
      s_kept_cnt[warp] = __popc(kb);
      s_pruned_cnt[warp] = __popc(pb);
    }
    __syncthreads();
    int kept_off = 0, pruned_off = 0, kept_total = 0, pruned_total = 0;
#pragma unroll
    for (int w = 0; w < PACK_WARPS; ++w) {
      const int kc = s_kept_cnt[w], pc = s_pruned_cnt[w];
      if (w < warp) { kept_off += kc; pruned_off += pc; }
      kept_total += kc;
      pruned_total += pc;
    }
    const int local_rank = kept_off + __popc(kb & lt_mask);
    const int excl = running + local_rank;   // kept tokens before g
    if (valid) {
      a.dst_idx[g] = kept ? excl : -1;
      if (kept) {
        a.src_idx[excl] = static_cast<int32_t>(g);
        long long srow = g;
        if (a.src_rows != nullptr) {
          srow = __ldg(a.src_rows + g);
          if (srow < 0 || srow >= a.src_cap) {   // kept now, pruned before: nothing to copy
            record_error(a.err, RRA_DEVERR_INDEX_RANGE);
            srow = -1;
          }
        }
        if (a.rows_out != nullptr) a.rows_out[excl] = static_cast<int32_t>(srow);
        s_kept_src[local_rank] = srow;
        s_kept_dst[local_rank] = excl;
      } else {
        s_pruned_g[pruned_off + __popc(pb & lt_mask)] = static_cast<int>(g - g0);
      }
      if (g % a.N == 0) a.cu_seqlens[g / a.N] = excl;
      if (g == total - 1) a.cu_seqlens[a.B] = excl + (kept ? 1 : 0);
    }
    __syncthreads();

    // Gather the kept rows: item = (kept token, 16-byte vector of its row).
    const int rv = a.row_vecs;
    const int items = kept_total * rv;
    int it = threadIdx.x;
    if (a.src_rows == nullptr) {
      for (; it + PACK_THREADS < items; it += 2 * PACK_THREADS) {
        const int t0 = it / rv, c0 = it - t0 * rv;
        const int i1 = it + PACK_THREADS;
        const int t1 = i1 / rv, c1 = i1 - t1 * rv;
        const size_t s0 = static_cast<size_t>(s_kept_src[t0]) * rv + c0;
        const size_t d0 = static_cast<size_t>(s_kept_dst[t0]) * rv + c0;
        const size_t s1 = static_cast<size_t>(s_kept_src[t1]) * rv + c1;
        const size_t d1 = static_cast<size_t>(s_kept_dst[t1]) * rv + c1;
        const uint4 q0 = __ldg(a.q + s0), k0 = __ldg(a.k + s0), v0 = __ldg(a.v + s0);
        const uint4 q1 = __ldg(a.q + s1), k1 = __ldg(a.k + s1), v1 = __ldg(a.v + s1);
        a.qp[d0] = q0; a.kp[d0] = k0; a.vp[d0] = v0;
        a.qp[d1] = q1; a.kp[d1] = k1; a.vp[d1] = v1;
      }
    }
    for (; it < items; it += PACK_THREADS) {
      const int t0 = it / rv, c0 = it - t0 * rv;
      const long long sr = s_kept_src[t0];
      if (sr < 0) continue;
      const size_t s0 = static_cast<size_t>(sr) * rv + c0;
      const size_t d0 = static_cast<size_t>(s_kept_dst[t0]) * rv + c0;
      const uint4 q0 = __ldg(a.q + s0), k0 = __ldg(a.k + s0), v0 = __ldg(a.v + s0);
      a.qp[d0] = q0; a.kp[d0] = k0; a.vp[d0] = v0;
    }

    // Zero the output rows of pruned tokens (the unpack's fill).
    if (a.out_zero != nullptr) {
      const int ov = a.out_row_vecs;
      const int zitems = pruned_total * ov;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int zi = threadIdx.x; zi < zitems; zi += PACK_THREADS) {
        const int t0 = zi / ov, c0 = zi - t0 * ov;
        a.out_zero[static_cast<size_t>(g0 + s_pruned_g[t0]) * ov + c0] = z;
      }
    }
    running += kept_total;
    __syncthreads();
  }
}

cudaError_t launch_pack(const PackArgs& a, int num_sms, cudaStream_t stream) {
  const long long total = static_cast<long long>(a.B) * a.N;
  PackArgs args = a;
  // A few CTAs per SM: enough memory parallelism for the gather while the
  // redundant prefix counting (each CTA reads keep[0, g0)) stays small.
  const long long target_ctas = 4LL * (num_sms > 0 ? num_sms : 152);
  long long tpc = (total + target_ctas - 1) / target_ctas;
  tpc = ((tpc + 31) / 32) * 32;
  if (tpc < 32) tpc = 32;
  args.tok_per_cta = static_cast<int>(tpc);
  const long long grid = (total + tpc - 1) / tpc;
  // A plain launch: as a programmatic dependent of a persistent attention
  // grid, the copy's CTAs took the SMs in the order that grid's CTAs
  // finished and ran unevenly (+17 us over the 12-layer chain with copies).
  pack_kernel<<<static_cast<unsigned>(grid), PACK_THREADS, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace rra

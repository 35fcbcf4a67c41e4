/* Second CPU oracle (test infrastructure only; the product never loads it):
 * the same definitions as oracle/ragged_attention.py, written again as plain
 * C loops in fp64, for tiny cases.  It is built by oracle/build_c.py and
 * called only by tests/test_oracle_c.py.
 *
 * Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers":
 * the agents-report.net article, section 方法概覽 (method overview), bullet 1
 * (per-image offsets cu_seqlens and destination indices of the kept tokens,
 * images in batch order, tokens in their original order) and bullet 2
 * (attention among each image's kept tokens only); the abstract (both
 * revisions) for the bidirectional (unmasked) attention over the pruned
 * sequence. */
#include <math.h>
#include <stdint.h>

/* cu_seqlens [B+1], dst_idx [B*N] (-1 where pruned), src_idx [T]. */
void rra_oracle_pack_indices(const uint8_t* keep, int B, int N, int32_t* cu, int32_t* dst, int32_t* src) {
  int t = 0;
  for (int b = 0; b < B; ++b) {
    cu[b] = t;
    for (int j = 0; j < N; ++j) {
      const int g = b * N + j;
      if (keep[g] != 0) {
        dst[g] = t;
        src[t] = g;
        ++t;
      } else {
        dst[g] = -1;
      }
    }
  }
  cu[B] = t;
}

/* o[i, h, :] = sum_j softmax_j(scale * <q[i,h,:], k[j,h,:]>) v[j, h, :] over
 * the rows j of row i's image; q, k, v, o packed [T, H, d], row-major. */
void rra_oracle_attend(const double* q, const double* k, const double* v, const int32_t* cu, int B, int H, int d,
                       double scale, double* o) {
  for (int b = 0; b < B; ++b) {
    const int s0 = cu[b], s1 = cu[b + 1];
    for (int h = 0; h < H; ++h) {
      for (int i = s0; i < s1; ++i) {
        const double* qi = q + ((long)i * H + h) * d;
        double m = -INFINITY;
        for (int j = s0; j < s1; ++j) {
          const double* kj = k + ((long)j * H + h) * d;
          double s = 0.0;
          for (int c = 0; c < d; ++c) s += qi[c] * kj[c];
          s *= scale;
          if (s > m) m = s;
        }
        double l = 0.0;
        double* oi = o + ((long)i * H + h) * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (int j = s0; j < s1; ++j) {
          const double* kj = k + ((long)j * H + h) * d;
          const double* vj = v + ((long)j * H + h) * d;
          double s = 0.0;
          for (int c = 0; c < d; ++c) s += qi[c] * kj[c];
          const double p = exp(s * scale - m);
          l += p;
          for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
        }
        for (int c = 0; c < d; ++c) oi[c] /= l;
      }
    }
  }
}

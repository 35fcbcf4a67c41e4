// Internal declarations shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/rra.h"

namespace rra {

inline int dtype_bytes(rra_dtype t) { return t == RRA_F32 ? 4 : 2; }

// Records a device-side error code: the first code wins, later ones are kept
// out so the reported code names the earliest anomaly seen.
__device__ __forceinline__ void record_error(int32_t* err, int32_t code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

struct PackArgs {
  const uint8_t* keep;
  int B, N;
  int tok_per_cta;    // tokens handled by one CTA (multiple of 32)
  int row_vecs;       // 16-byte vectors per token row of q/k/v (H*d*in_bytes/16)
  int out_row_vecs;   // 16-byte vectors per token row of the zero-filled output, 0 = none
  const uint4* q;
  const uint4* k;
  const uint4* v;
  uint4* qp;
  uint4* kp;
  uint4* vp;
  uint4* out_zero;
  int32_t* cu_seqlens;
  int32_t* dst_idx;
  int32_t* src_idx;
  // Re-pack: the row copied for kept position g is row src_rows[g] of q/k/v
  // (a previous layer's packed buffers, src_cap rows) instead of row g.
  const int32_t* src_rows;
  long long src_cap;
  // Optional: rows_out[t] = the row copied (or, with row_vecs == 0, to be
  // read) for packed row t: src_rows[g], or g itself without src_rows.
  int32_t* rows_out;
  int32_t* err;
};

struct AttendArgs {
  const uint8_t* keep;      // fused pipeline only: the mask, scanned on the device
  const void* qp;
  const void* kp;
  const void* vp;
  const int32_t* cu_seqlens;
  const int32_t* src_idx;   // nullptr: packed output
  void* o;
  int B, H, N, max_seqlen;
  float scale_log2;         // softmax scale times log2(e)
  int32_t* err;
  // Completion signal for a host that polls instead of synchronising the
  // stream (rra_attend_wait); done_count == nullptr: off.
  uint32_t* done_count;     // count of finished CTAs, never reset: a device word,
                            // or (done_word == nullptr) a page-locked host word
  uint32_t done_target;     // its value before this launch (the launcher adds the grid size)
  uint32_t* done_word;      // device address of a page-locked host word, or nullptr
  uint32_t done_ticket;     // value published to *done_word
  long long wait_limit;     // clock cycles one on-chip wait may take before giving up (0: the default)
  // Row-gather inputs with a packed output (launch_attend_tc_rows): q/k/v
  // span src_rows rows and packed row t is read from row src_idx[t].
  // 0: the padded gather (B*N rows, output scattered to src_idx).
  long long src_rows;
  // Class-token side output (launches with a CLS instantiation only): cls
  // [B, H, cls_stride] fp32 receives, for every image's first row, its
  // softmax weights over the image's rows (see rra_attend_cls).
  float* cls;
  int cls_stride;
};

// Each CTA adds one to *done_count once all its threads' output stores are
// issued, with release semantics, so by cumulativity every CTA's stores are
// visible before the count moves.  The count is never reset and no CTA waits
// on another.  Two forms:
//   done_word == nullptr: the count is itself a page-locked host word (the
//     device has native atomics on host memory); each CTA adds with a
//     system-scope release reduction, no round trip, and the host polls the
//     count until it reaches done_target.
//   otherwise: the count is a device word; the CTA whose add brings it to
//     done_target publishes done_ticket to the host word with a
//     system-scope release store.
// Called by all threads of the CTA (it holds a CTA barrier).  `wrote`: the
// CTA stored output; a CTA that stored nothing adds with a relaxed
// reduction (it has nothing to publish; the release sequence of the other
// CTAs' adds continues through it).
__device__ __forceinline__ void signal_done(const AttendArgs& a, bool wrote = true) {
  __syncthreads();
  if (threadIdx.x == 0) {
    if (a.done_word == nullptr) {
      if (wrote) asm volatile("red.release.sys.global.add.u32 [%0], 1;" ::"l"(a.done_count) : "memory");
      else asm volatile("red.relaxed.sys.global.add.u32 [%0], 1;" ::"l"(a.done_count) : "memory");
    } else {
      uint32_t prev;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(a.done_count) : "memory");
      if (prev + 1u == a.done_target)
        asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(a.done_word), "r"(a.done_ticket) : "memory");
    }
  }
}

struct UnpackArgs {
  const uint4* op;
  const int32_t* dst_idx;
  uint4* out;
  int B, N;
  int row_vecs;
  int32_t* err;
};

// Sets the message rra_last_error_message() returns on the calling thread.
void set_last_error_message(const char* msg);

// Launchers (each enqueues exactly one kernel on `stream`).
cudaError_t launch_pack(const PackArgs& a, int num_sms, cudaStream_t stream);
// The attention launchers add their grid size to a.done_target when a
// completion signal is on and report it through *ctas (when not null).
cudaError_t launch_attend(const AttendArgs& a, rra_dtype in, rra_dtype out, cudaStream_t stream,
                          uint32_t* ctas = nullptr);
cudaError_t launch_unpack(const UnpackArgs& a, cudaStream_t stream);
// Packed linear layer on the tensor cores: c[t] = a[t] W^T (+ bias) for the
// T = cu[B] kept rows (T read on the device).
cudaError_t launch_linear_packed(const void* a, const void* w, const float* bias, const int32_t* cu, int B,
                                 int cap, int K, int N, rra_dtype in, void* c, rra_dtype out, int32_t* err,
                                 cudaStream_t stream);
// Device-side pruning step: class-token attention scores [B, N] and the
// top-k keep decision (one CTA per image each).
cudaError_t launch_cls_scores(const void* qp, const void* kp, const int32_t* cu, const int32_t* src, int B, int N,
                              int H, float scale, rra_dtype in, float* scores, int32_t* err, cudaStream_t stream);
cudaError_t launch_topk_keep(const float* scores, const uint8_t* keep_prev, int B, int N, int num, int den,
                             uint8_t* keep_new, cudaStream_t stream);
// The keep decision from the attention's class-token side output cls
// [B, H, stride] (one CTA per image); keep_new and scores [B, N] optional;
// with cu_new (not null) also the next layer's cu/dst/src and rows.
cudaError_t launch_prune_cls(const float* cls, int stride, const int32_t* cu, const int32_t* src, int B, int N, int H,
                             int num, int den, uint8_t* keep_new, float* scores, int32_t* cu_new, int32_t* dst_new,
                             int32_t* src_new, int32_t* rows_new, int32_t* err, cudaStream_t stream);
// tcgen05 + TMA attention; needs the driver's tensor-map encoder.
bool attend_tc_available();
cudaError_t launch_attend_tc(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms, cudaStream_t stream,
                             uint32_t* ctas = nullptr);
// Same kernel reading Q/K/V rows straight from the padded [B, N, H, 64]
// tensors (a.qp/kp/vp) at rows src_idx[t], scattering to the padded output.
cudaError_t launch_attend_tc_gather(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                    cudaStream_t stream);
// Same kernel reading packed row t of Q/K/V from row a.src_idx[t] of the
// [a.src_rows, H, 64] buffers a.qp/kp/vp and writing the packed output row t.
cudaError_t launch_attend_tc_rows(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                  cudaStream_t stream);
// The whole pipeline in one launch: the same kernel scanning the keep mask
// per image, gathering from the padded q/k/v, writing every output row
// (attention at kept positions, +0 at pruned ones).  a.keep, a.qp/kp/vp
// (padded), a.o, a.B, a.N, a.H, a.scale_log2, a.err are used.
cudaError_t launch_attend_tc_fused(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                   cudaStream_t stream);
// Longest image (kept tokens) the small-grid kernel takes: its K and V rows
// stay in shared memory for the whole unit.
constexpr int ATTEND_SMALL_MAX_KEYS = 256;
// Small grids (about one unit per SM): one CTA of four warps per (image,
// head, query tile), no warp specialisation; max_seqlen <= 256.  fused:
// the whole pipeline (a.keep scanned, rows gathered from the padded
// a.qp/kp/vp, every output row written; a.max_seqlen == a.N); else packed
// inputs as launch_attend_tc.
cudaError_t launch_attend_small(const AttendArgs& a, rra_dtype in, rra_dtype out, bool fused, cudaStream_t stream,
                                uint32_t* ctas = nullptr);
// The same pipeline for keep/q/k/v/o in page-locked host memory (device
// addresses of the mapping): the rows come in by cp.async copies instead of
// TMA, every output row leaves by plain stores.
cudaError_t launch_attend_tc_fused_host(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                        cudaStream_t stream);

}  // namespace rra

// C-ABI entry points of librra (declared in include/rra.h): host-side
// argument checks, workspace layout, the two-launch pipeline, CUDA-graph
// plans, the device error word and host-timing helpers.
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace rra {
namespace {

// Device-side error word (one per device that loads the library).
__device__ int32_t g_device_error = 0;

__global__ void null_kernel() {}

thread_local char g_last_message[256] = "";
// rra_bind_error_word: the error word of this host thread's launches (null:
// the device's own word).
thread_local int32_t* g_bound_error_word = nullptr;
// rra_set_wait_limit: the attention kernels' bound on one on-chip wait, in
// clock cycles (0: the kernels' default).
std::atomic<long long> g_wait_limit{0};
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_attend_kernel{RRA_ATTEND_AUTO};


rra_status fail(rra_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_message, sizeof(g_last_message), fmt, ap);
  va_end(ap);
  return s;
}

rra_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RRA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// rra_attend_wait's count of finished CTAs (one per device, 0 between launches).
__device__ uint32_t g_done_count = 0;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int32_t* err = nullptr;
  // rra_attend_wait: the page-locked host word the last CTA publishes to,
  // made on first use, and the ticket of the latest call.  wait_mutex
  // serialises the calls on this device (they share the count and the word).
  std::mutex wait_mutex;
  bool host_count = false;     // the CTA count is the host word itself (native host atomics)
  uint32_t* done_count = nullptr;
  uint32_t* host_word = nullptr;
  uint32_t* host_word_dev = nullptr;
  uint32_t ticket = 0;
  uint32_t ctas_counted = 0;   // CTAs launched with a signal so far (mod 2^32)
};

constexpr int kMaxDevices = 64;
DeviceState g_devices[kMaxDevices];
std::mutex g_device_mutex;

// Per-device set-up, done once per device with that device current.
rra_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(RRA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  DeviceState& st = g_devices[dev];
  std::lock_guard<std::mutex> lock(g_device_mutex);
  if (!st.ready) {
    e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    st.err = static_cast<int32_t*>(p);
    st.ready = true;
  }
  *out = &st;
  return RRA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Where the kernels this thread enqueues record device-side errors.
int32_t* error_word(const DeviceState& st) { return g_bound_error_word != nullptr ? g_bound_error_word : st.err; }

bool valid_in(rra_dtype t) { return t == RRA_F16 || t == RRA_BF16; }
bool valid_out(rra_dtype t) { return t == RRA_F16 || t == RRA_BF16 || t == RRA_F32; }
bool finite(float x) { return x == x && x != INFINITY && x != -INFINITY; }

rra_status check_shape(int B, int N, int H, int d) {
  if (d != 64) return fail(RRA_ERR_UNSUPPORTED, "head dim %d unsupported (only 64)", d);
  if (B < 1 || B > 65535) return fail(RRA_ERR_INVALID_ARG, "B=%d outside [1, 65535]", B);
  if (N < 1) return fail(RRA_ERR_INVALID_ARG, "N=%d < 1", N);
  if (N > 1024) return fail(RRA_ERR_UNSUPPORTED, "N=%d > 1024", N);
  if (H < 1 || H > 65535) return fail(RRA_ERR_INVALID_ARG, "H=%d outside [1, 65535]", H);
  const long long elems = static_cast<long long>(B) * N * H * d;
  if (elems >= (1LL << 31)) return fail(RRA_ERR_UNSUPPORTED, "B*N*H*d=%lld >= 2^31", elems);
  return RRA_OK;
}

#define RRA_CHECK_PTR(p)                                                               \
  do {                                                                                 \
    if ((p) == nullptr) return fail(RRA_ERR_INVALID_ARG, "%s is null", #p);           \
    if (!aligned16(p)) return fail(RRA_ERR_MISALIGNED, "%s not 16-byte aligned", #p); \
  } while (0)

#define RRA_TRY(expr)            \
  do {                           \
    rra_status _s = (expr);      \
    if (_s != RRA_OK) return _s; \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

void workspace_layout(int B, int N, int H, int d, rra_dtype in, size_t off[6], size_t* total) {
  const size_t tokens = static_cast<size_t>(B) * N;
  const size_t packed = tokens * H * d * dtype_bytes(in);
  size_t o = 0;
  off[0] = o; o = align256(o + (static_cast<size_t>(B) + 1) * 4);
  off[1] = o; o = align256(o + tokens * 4);
  off[2] = o; o = align256(o + tokens * 4);
  off[3] = o; o = align256(o + packed);
  off[4] = o; o = align256(o + packed);
  off[5] = o; o = align256(o + packed);
  *total = o;
}

// ---------------------------------------------------------------- enqueue

// The attention kernel a call runs under the current choice: the
// warp-specialised tcgen05 kernel, its small-grid form (one warpgroup per
// unit, max_seqlen <= 256), or the mma.sync kernel.
enum AttendKernelChoice { KC_TC = 0, KC_TC_SMALL = 1, KC_MMA = 2 };
AttendKernelChoice attend_choice(const DeviceState& st, int B, int H, int max_seqlen, bool pipeline) {
  const int k = g_attend_kernel.load();
  const bool small_ok = max_seqlen <= ATTEND_SMALL_MAX_KEYS;
  if (k == RRA_ATTEND_MMA_SYNC) return KC_MMA;
  if (k == RRA_ATTEND_TCGEN05) return KC_TC;
  if (k == RRA_ATTEND_TCGEN05_LATENCY) return small_ok ? KC_TC_SMALL : KC_TC;
  // Automatic.  While the grid has a few units per SM each CTA is mostly
  // one latency chain: the pipeline takes the small-grid tcgen05 form (one
  // launch that also scans the mask and writes the zero rows) up to four
  // units per SM (serving-like batches, N=197, H=6, fused us small / warp-
  // specialised: B=4 4.0 / 5.3, B=32 5.8 / 6.7, B=48 7.1 / 7.4, B=64
  // 10.1 / 8.3), rra_attend on packed buffers the mma.sync kernel up to two
  // (its register-resident chain returns to a polling host in 10.2-10.4 us
  // against 10.6-10.7 us at B=1-4).  Beyond, the warp-specialised kernel.
  const long long units = static_cast<long long>(B) * H * ((max_seqlen + 127) / 128);
  if (small_ok && pipeline && units <= 4LL * st.num_sms) return KC_TC_SMALL;
  if (small_ok && !pipeline && units <= 2LL * st.num_sms) return KC_MMA;
  return KC_TC;
}

rra_status enqueue_pack(const DeviceState& st, const uint8_t* keep, int B, int N, int H, int d,
                        rra_dtype in, const void* q, const void* k, const void* v, int32_t* cu,
                        int32_t* dst, int32_t* src, void* qp, void* kp, void* vp, void* outz,
                        rra_dtype out_dt, cudaStream_t s, const int32_t* src_rows = nullptr,
                        int32_t* rows_out = nullptr) {
  PackArgs a{};
  a.src_rows = src_rows;
  a.rows_out = rows_out;
  a.src_cap = static_cast<long long>(B) * N;
  a.err = error_word(st);
  a.keep = keep;
  a.B = B;
  a.N = N;
  a.row_vecs = (qp != nullptr) ? H * d * dtype_bytes(in) / 16 : 0;   // 0: indices and zero fill only
  a.out_row_vecs = outz ? H * d * dtype_bytes(out_dt) / 16 : 0;
  a.q = static_cast<const uint4*>(q);
  a.k = static_cast<const uint4*>(k);
  a.v = static_cast<const uint4*>(v);
  a.qp = static_cast<uint4*>(qp);
  a.kp = static_cast<uint4*>(kp);
  a.vp = static_cast<uint4*>(vp);
  a.out_zero = static_cast<uint4*>(outz);
  a.cu_seqlens = cu;
  a.dst_idx = dst;
  a.src_idx = src;
  cudaError_t e = launch_pack(a, st.num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "pack launch");
  return RRA_OK;
}

rra_status check_attend(const void* qp, const void* kp, const void* vp, const int32_t* cu_seqlens, int B,
                        int max_seqlen, int H, int d, float scale, rra_dtype in_dtype, const void* o,
                        rra_dtype out_dtype, const int32_t* src_idx, int N) {
  RRA_TRY(check_shape(B, max_seqlen, H, d));
  if (!valid_in(in_dtype)) return fail(RRA_ERR_INVALID_ARG, "input dtype invalid");
  if (!valid_out(out_dtype)) return fail(RRA_ERR_INVALID_ARG, "output dtype invalid");
  if (!finite(scale)) return fail(RRA_ERR_INVALID_ARG, "scale is not finite");
  RRA_CHECK_PTR(qp);
  RRA_CHECK_PTR(kp);
  RRA_CHECK_PTR(vp);
  RRA_CHECK_PTR(o);
  if (cu_seqlens == nullptr) return fail(RRA_ERR_INVALID_ARG, "cu_seqlens is null");
  if (src_idx != nullptr) RRA_TRY(check_shape(B, N, H, d));
  return RRA_OK;
}

// The page-locked host word and device count of rra_attend_wait, made on
// first use (caller holds st.wait_mutex).
rra_status done_signal_state(DeviceState& st) {
  if (st.host_word != nullptr) return RRA_OK;
  void* h = nullptr;
  cudaError_t e = cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc(completion word)");
  void* dp = nullptr;
  e = cudaHostGetDevicePointer(&dp, h, 0);
  void* cnt = nullptr;
  if (e == cudaSuccess) e = cudaGetSymbolAddress(&cnt, g_done_count);
  if (e != cudaSuccess) {
    cudaFreeHost(h);
    return cuda_fail(e, "completion word mapping");
  }
  int dev = 0, native = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&native, cudaDevAttrHostNativeAtomicSupported, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    native = 0;
  }
  __atomic_store_n(static_cast<uint32_t*>(h), 0u, __ATOMIC_RELEASE);
  st.host_word = static_cast<uint32_t*>(h);
  st.host_word_dev = static_cast<uint32_t*>(dp);
  // RRA_WAIT_DEVICE_COUNT=1 selects the device-word form even where host
  // atomics are native (so both forms can be exercised on one machine).
  const char* force = getenv("RRA_WAIT_DEVICE_COUNT");
  st.host_count = native != 0 && !(force != nullptr && force[0] == '1');
  // With native host atomics the CTAs count straight into the host word;
  // otherwise into a device word, and the last CTA publishes a ticket.
  st.done_count = st.host_count ? st.host_word_dev : static_cast<uint32_t*>(cnt);
  st.ctas_counted = 0;
  return RRA_OK;
}

struct DoneSignal {
  uint32_t* count;
  uint32_t count_base;   // *count before this launch
  uint32_t* word;
  uint32_t ticket;
};

rra_status enqueue_attend(const DeviceState& st, const void* qp, const void* kp, const void* vp,
                          const int32_t* cu, int B, int max_seqlen, int H, float scale,
                          rra_dtype in, void* o, rra_dtype out_dt, const int32_t* src_idx, int N,
                          cudaStream_t s, const DoneSignal* done = nullptr, uint32_t* ctas = nullptr,
                          bool coalesced_out = false) {
  AttendArgs a{};
  if (done != nullptr) {
    a.done_count = done->count;
    a.done_target = done->count_base;
    a.done_word = done->word;
    a.done_ticket = done->ticket;
  }
  a.qp = qp;
  a.kp = kp;
  a.vp = vp;
  a.cu_seqlens = cu;
  a.src_idx = src_idx;
  a.o = o;
  a.B = B;
  a.H = H;
  a.N = N;
  a.max_seqlen = max_seqlen;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = error_word(st);
  a.wait_limit = g_wait_limit.load();
  cudaError_t e;
  const AttendKernelChoice kc = coalesced_out ? KC_MMA : attend_choice(st, B, H, max_seqlen, false);
  if (kc == KC_TC) {
    if (!attend_tc_available())
      return fail(RRA_ERR_CUDA, "attend: the driver's tensor-map encoder is unavailable");
    e = launch_attend_tc(a, in, out_dt, st.num_sms, s, ctas);
  } else if (kc == KC_TC_SMALL) {
    e = launch_attend_small(a, in, out_dt, false, s, ctas);
  } else {
    e = launch_attend(a, in, out_dt, s, ctas);
  }
  if (e != cudaSuccess) return cuda_fail(e, "attend launch");
  return RRA_OK;
}

struct PipelineArgs {
  const uint8_t* keep;
  const void *q, *k, *v;
  int B, N, H, d;
  float scale;
  rra_dtype in, out_dt;
  void* out;
  void* ws;
  size_t ws_bytes;
};

rra_status check_pipeline(const PipelineArgs& p) {
  RRA_TRY(check_shape(p.B, p.N, p.H, p.d));
  if (!valid_in(p.in)) return fail(RRA_ERR_INVALID_ARG, "input dtype %d invalid", static_cast<int>(p.in));
  if (!valid_out(p.out_dt))
    return fail(RRA_ERR_INVALID_ARG, "output dtype %d invalid", static_cast<int>(p.out_dt));
  if (!finite(p.scale)) return fail(RRA_ERR_INVALID_ARG, "scale is not finite");
  if (p.keep == nullptr) return fail(RRA_ERR_INVALID_ARG, "keep is null");
  RRA_CHECK_PTR(p.q);
  RRA_CHECK_PTR(p.k);
  RRA_CHECK_PTR(p.v);
  RRA_CHECK_PTR(p.out);
  RRA_CHECK_PTR(p.ws);
  size_t off[6], total = 0;
  workspace_layout(p.B, p.N, p.H, p.d, p.in, off, &total);
  if (p.ws_bytes < total)
    return fail(RRA_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", p.ws_bytes, total);
  return RRA_OK;
}

// rra_pipeline's choice: the fused one-launch tcgen05 kernel unless the
// mma.sync kernel was selected explicitly (one launch beats pack + attend
// even where the batch is too small to fill the GPU).
bool pipeline_fused() { return g_attend_kernel.load() != RRA_ATTEND_MMA_SYNC; }

// Kernel launches one rra_pipeline call makes: 1 fused, 2 packed.
int pipeline_launches(const DeviceState&, const PipelineArgs&) { return pipeline_fused() ? 1 : 2; }

// The two-launch form: rra_pack (with the row copy, and the zero fill of the
// pruned output rows) into the workspace, then rra_attend on the packed
// buffers scattering to the padded output.  coalesced_out: the output is in
// host memory; take the mma.sync attention, whose epilogue writes whole
// 128-byte lines per store instruction (the tcgen05 epilogue writes one row
// per thread, which crosses the link as partial lines: 213 against 142 us on
// B=64 at 80% pruning).
rra_status enqueue_packed_pipeline(const DeviceState& st, const PipelineArgs& p, cudaStream_t s,
                                   bool coalesced_out = false) {
  size_t off[6], total = 0;
  workspace_layout(p.B, p.N, p.H, p.d, p.in, off, &total);
  uint8_t* ws = static_cast<uint8_t*>(p.ws);
  int32_t* cu = reinterpret_cast<int32_t*>(ws + off[0]);
  int32_t* dst = reinterpret_cast<int32_t*>(ws + off[1]);
  int32_t* src = reinterpret_cast<int32_t*>(ws + off[2]);
  void* qp = ws + off[3];
  void* kp = ws + off[4];
  void* vp = ws + off[5];
  RRA_TRY(enqueue_pack(st, p.keep, p.B, p.N, p.H, p.d, p.in, p.q, p.k, p.v, cu, dst, src, qp, kp, vp,
                       p.out, p.out_dt, s));
  return enqueue_attend(st, qp, kp, vp, cu, p.B, p.N, p.H, p.scale, p.in, p.out, p.out_dt, src, p.N, s, nullptr,
                        nullptr, coalesced_out);
}

rra_status enqueue_pipeline(const DeviceState& st, const PipelineArgs& p, cudaStream_t s) {
  if (pipeline_fused()) {
    // One launch: the attention kernel scans the keep mask per image,
    // gathers the kept rows straight from q/k/v and writes every output row.
    if (!attend_tc_available())
      return fail(RRA_ERR_CUDA, "pipeline: the driver's tensor-map encoder is unavailable");
    AttendArgs a{};
    a.keep = p.keep;
    a.qp = p.q;
    a.kp = p.k;
    a.vp = p.v;
    a.o = p.out;
    a.B = p.B;
    a.H = p.H;
    a.N = p.N;
    a.max_seqlen = p.N;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.err = error_word(st);
    a.wait_limit = g_wait_limit.load();
    cudaError_t e = attend_choice(st, p.B, p.H, p.N, true) == KC_TC_SMALL
                        ? launch_attend_small(a, p.in, p.out_dt, true, s)
                        : launch_attend_tc_fused(a, p.in, p.out_dt, st.num_sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "fused pipeline launch");
    return RRA_OK;
  }
  return enqueue_packed_pipeline(st, p, s);
}

// The address through which the current device reaches page-locked host
// memory at p (cudaHostAlloc / cudaMallocHost / cudaHostRegister), or null
// for anything else (pageable, device or managed memory).
void* mapped_host_ptr(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

bool is_device_memory(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice;
}

}  // namespace

void set_last_error_message(const char* msg) {
  snprintf(g_last_message, sizeof(g_last_message), "%s", msg);
}

}  // namespace rra

using namespace rra;

struct rra_plan {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int launches = 0;
};

extern "C" {

const char* rra_status_string(rra_status s) {
  switch (s) {
    case RRA_OK: return "RRA_OK";
    case RRA_ERR_INVALID_ARG: return "RRA_ERR_INVALID_ARG";
    case RRA_ERR_UNSUPPORTED: return "RRA_ERR_UNSUPPORTED";
    case RRA_ERR_MISALIGNED: return "RRA_ERR_MISALIGNED";
    case RRA_ERR_CUDA: return "RRA_ERR_CUDA";
    case RRA_ERR_DEVICE: return "RRA_ERR_DEVICE";
  }
  return "RRA_UNKNOWN_STATUS";
}

const char* rra_last_error_message(void) { return g_last_message; }

uint64_t rra_launch_count(void) { return g_launches.load(); }

int rra_set_attend_kernel(int kernel) {
  if (kernel != RRA_ATTEND_TCGEN05 && kernel != RRA_ATTEND_MMA_SYNC && kernel != RRA_ATTEND_AUTO &&
      kernel != RRA_ATTEND_TCGEN05_LATENCY)
    return -1;
  return g_attend_kernel.exchange(kernel);
}

size_t rra_workspace_bytes(int B, int N, int H, int d, rra_dtype in_dtype) {
  if (check_shape(B, N, H, d) != RRA_OK || !valid_in(in_dtype)) return 0;
  size_t off[6], total = 0;
  workspace_layout(B, N, H, d, in_dtype, off, &total);
  return total;
}

rra_status rra_workspace_offsets(int B, int N, int H, int d, rra_dtype in_dtype, size_t offsets[6]) {
  RRA_TRY(check_shape(B, N, H, d));
  if (!valid_in(in_dtype)) return fail(RRA_ERR_INVALID_ARG, "input dtype invalid");
  if (offsets == nullptr) return fail(RRA_ERR_INVALID_ARG, "offsets is null");
  size_t total = 0;
  workspace_layout(B, N, H, d, in_dtype, offsets, &total);
  return RRA_OK;
}

rra_status rra_pack(const uint8_t* keep, int B, int N, int H, int d, rra_dtype in_dtype,
                    const void* q, const void* k, const void* v, int32_t* cu_seqlens,
                    int32_t* dst_idx, int32_t* src_idx, void* qp, void* kp, void* vp,
                    void* out_zero_fill, rra_dtype out_dtype, void* stream) {
  RRA_TRY(check_shape(B, N, H, d));
  if (!valid_in(in_dtype)) return fail(RRA_ERR_INVALID_ARG, "input dtype invalid");
  if (out_zero_fill && !valid_out(out_dtype)) return fail(RRA_ERR_INVALID_ARG, "output dtype invalid");
  if (keep == nullptr) return fail(RRA_ERR_INVALID_ARG, "keep is null");
  const bool index_only = (qp == nullptr && kp == nullptr && vp == nullptr);
  if (!index_only) {
    RRA_CHECK_PTR(q);
    RRA_CHECK_PTR(k);
    RRA_CHECK_PTR(v);
    RRA_CHECK_PTR(qp);
    RRA_CHECK_PTR(kp);
    RRA_CHECK_PTR(vp);
  }
  if (cu_seqlens == nullptr || dst_idx == nullptr || src_idx == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "index buffer is null");
  if (out_zero_fill && !aligned16(out_zero_fill))
    return fail(RRA_ERR_MISALIGNED, "out_zero_fill not 16-byte aligned");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  RRA_TRY(enqueue_pack(*st, keep, B, N, H, d, in_dtype, q, k, v, cu_seqlens, dst_idx, src_idx, qp, kp, vp,
                       out_zero_fill, out_dtype, static_cast<cudaStream_t>(stream)));
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_repack(const uint8_t* keep_new, const int32_t* dst_prev, int B, int N, int H, int d,
                      rra_dtype in_dtype, const void* qp_prev, const void* kp_prev, const void* vp_prev,
                      int32_t* cu_seqlens, int32_t* dst_idx, int32_t* src_idx, void* qp, void* kp, void* vp,
                      void* stream) {
  RRA_TRY(check_shape(B, N, H, d));
  if (!valid_in(in_dtype)) return fail(RRA_ERR_INVALID_ARG, "input dtype invalid");
  if (keep_new == nullptr || dst_prev == nullptr) return fail(RRA_ERR_INVALID_ARG, "keep_new or dst_prev is null");
  RRA_CHECK_PTR(qp_prev);
  RRA_CHECK_PTR(kp_prev);
  RRA_CHECK_PTR(vp_prev);
  RRA_CHECK_PTR(qp);
  RRA_CHECK_PTR(kp);
  RRA_CHECK_PTR(vp);
  if (cu_seqlens == nullptr || dst_idx == nullptr || src_idx == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "index buffer is null");
  const size_t bytes = static_cast<size_t>(B) * N * H * d * dtype_bytes(in_dtype);
  const void* prev[3] = {qp_prev, kp_prev, vp_prev};
  const void* next[3] = {qp, kp, vp};
  for (const void* x : prev)
    for (const void* y : next) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(x), b0 = reinterpret_cast<uintptr_t>(y);
      if (a0 < b0 + bytes && b0 < a0 + bytes) return fail(RRA_ERR_INVALID_ARG, "previous and new packed buffers overlap");
    }
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  RRA_TRY(enqueue_pack(*st, keep_new, B, N, H, d, in_dtype, qp_prev, kp_prev, vp_prev, cu_seqlens, dst_idx, src_idx,
                       qp, kp, vp, nullptr, RRA_F32, static_cast<cudaStream_t>(stream), dst_prev));
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_pack_index(const uint8_t* keep, const int32_t* dst_prev, int B, int N, int32_t* cu_seqlens,
                          int32_t* dst_idx, int32_t* src_idx, int32_t* rows, void* stream) {
  RRA_TRY(check_shape(B, N, 1, 64));
  if (keep == nullptr) return fail(RRA_ERR_INVALID_ARG, "keep is null");
  if (cu_seqlens == nullptr || dst_idx == nullptr || src_idx == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "index buffer is null");
  if (dst_prev != nullptr && dst_prev == dst_idx) return fail(RRA_ERR_INVALID_ARG, "dst_prev is dst_idx");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  RRA_TRY(enqueue_pack(*st, keep, B, N, 1, 64, RRA_BF16, nullptr, nullptr, nullptr, cu_seqlens, dst_idx, src_idx,
                       nullptr, nullptr, nullptr, nullptr, RRA_F32, static_cast<cudaStream_t>(stream), dst_prev, rows));
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_topk_keep_cls(const float* cls, int cls_stride, const int32_t* cu_seqlens, const int32_t* src_idx,
                             int B, int N, int H, int keep_num, int keep_den, uint8_t* keep_new, float* scores,
                             void* stream) {
  RRA_TRY(check_shape(B, N, H, 64));
  if (cls == nullptr || cu_seqlens == nullptr || src_idx == nullptr || keep_new == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "a required buffer is null");
  if (cls_stride < N) return fail(RRA_ERR_INVALID_ARG, "cls_stride=%d < N=%d", cls_stride, N);
  if (static_cast<long long>(B) * H * cls_stride >= (1LL << 31)) return fail(RRA_ERR_UNSUPPORTED, "cls too large");
  if (keep_den < 1 || keep_num < 0 || keep_num > keep_den)
    return fail(RRA_ERR_INVALID_ARG, "keep fraction %d/%d outside [0, 1]", keep_num, keep_den);
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaError_t e = launch_prune_cls(cls, cls_stride, cu_seqlens, src_idx, B, N, H, keep_num, keep_den, keep_new, scores,
                                   nullptr, nullptr, nullptr, nullptr, error_word(*st),
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "topk_keep_cls launch");
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_prune_index(const float* cls, int cls_stride, const int32_t* cu_prev, const int32_t* src_prev, int B,
                           int N, int H, int keep_num, int keep_den, int32_t* cu_seqlens, int32_t* dst_idx,
                           int32_t* src_idx, int32_t* rows, uint8_t* keep_new, float* scores, void* stream) {
  RRA_TRY(check_shape(B, N, H, 64));
  if (cls == nullptr || cu_prev == nullptr || src_prev == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "cls, cu_prev or src_prev is null");
  if (cu_seqlens == nullptr || dst_idx == nullptr || src_idx == nullptr || rows == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "index buffer is null");
  if (cu_seqlens == cu_prev || src_idx == src_prev) return fail(RRA_ERR_INVALID_ARG, "new and previous indices alias");
  if (cls_stride < N) return fail(RRA_ERR_INVALID_ARG, "cls_stride=%d < N=%d", cls_stride, N);
  if (static_cast<long long>(B) * H * cls_stride >= (1LL << 31)) return fail(RRA_ERR_UNSUPPORTED, "cls too large");
  if (keep_den < 1 || keep_num < 0 || keep_num > keep_den)
    return fail(RRA_ERR_INVALID_ARG, "keep fraction %d/%d outside [0, 1]", keep_num, keep_den);
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaError_t e = launch_prune_cls(cls, cls_stride, cu_prev, src_prev, B, N, H, keep_num, keep_den, keep_new, scores,
                                   cu_seqlens, dst_idx, src_idx, rows, error_word(*st),
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prune_index launch");
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_linear_packed(const void* a, const void* w, const float* bias, const int32_t* cu_seqlens, int B,
                             int cap, int K, int N, rra_dtype in_dtype, void* c, rra_dtype out_dtype,
                             void* stream) {
  if (B < 1 || B > 65535) return fail(RRA_ERR_INVALID_ARG, "B=%d outside [1, 65535]", B);
  if (cap < 1 || cap > 65535 * 128) return fail(RRA_ERR_INVALID_ARG, "cap=%d outside [1, 65535*128]", cap);
  if (K < 64 || K % 64 != 0 || K > 16384) return fail(RRA_ERR_UNSUPPORTED, "K=%d: a multiple of 64 up to 16384", K);
  if (N < 128 || N % 128 != 0 || N > 65535 * 128)
    return fail(RRA_ERR_UNSUPPORTED, "N=%d: a multiple of 128", N);
  if (!valid_in(in_dtype)) return fail(RRA_ERR_INVALID_ARG, "input dtype invalid");
  if (!valid_out(out_dtype)) return fail(RRA_ERR_INVALID_ARG, "output dtype invalid");
  RRA_CHECK_PTR(a);
  RRA_CHECK_PTR(w);
  RRA_CHECK_PTR(c);
  if (cu_seqlens == nullptr) return fail(RRA_ERR_INVALID_ARG, "cu_seqlens is null");
  if (bias != nullptr && !aligned16(bias)) return fail(RRA_ERR_MISALIGNED, "bias not 16-byte aligned");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaError_t e = launch_linear_packed(a, w, bias, cu_seqlens, B, cap, K, N, in_dtype, c, out_dtype, error_word(*st),
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "linear_packed launch");
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_cls_scores(const void* qp, const void* kp, const int32_t* cu_seqlens, const int32_t* src_idx,
                          int B, int N, int H, int d, float scale, rra_dtype in_dtype, float* scores,
                          void* stream) {
  RRA_TRY(check_shape(B, N, H, d));
  if (!valid_in(in_dtype)) return fail(RRA_ERR_INVALID_ARG, "input dtype invalid");
  if (!finite(scale)) return fail(RRA_ERR_INVALID_ARG, "scale is not finite");
  RRA_CHECK_PTR(qp);
  RRA_CHECK_PTR(kp);
  if (cu_seqlens == nullptr || src_idx == nullptr || scores == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "cu_seqlens, src_idx or scores is null");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaError_t e = launch_cls_scores(qp, kp, cu_seqlens, src_idx, B, N, H, scale, in_dtype, scores, error_word(*st),
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cls_scores launch");
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_topk_keep(const float* scores, const uint8_t* keep_prev, int B, int N, int keep_num, int keep_den,
                         uint8_t* keep_new, void* stream) {
  RRA_TRY(check_shape(B, N, 1, 64));
  if (scores == nullptr || keep_prev == nullptr || keep_new == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "scores, keep_prev or keep_new is null");
  if (keep_den < 1 || keep_num < 0 || keep_num > keep_den)
    return fail(RRA_ERR_INVALID_ARG, "keep fraction %d/%d outside [0, 1]", keep_num, keep_den);
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(keep_prev), b0 = reinterpret_cast<uintptr_t>(keep_new);
  const size_t bytes = static_cast<size_t>(B) * N;
  if (a0 < b0 + bytes && b0 < a0 + bytes) return fail(RRA_ERR_INVALID_ARG, "keep_prev and keep_new overlap");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaError_t e = launch_topk_keep(scores, keep_prev, B, N, keep_num, keep_den, keep_new,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "topk_keep launch");
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_attend(const void* qp, const void* kp, const void* vp, const int32_t* cu_seqlens,
                      int B, int max_seqlen, int H, int d, float scale, rra_dtype in_dtype, void* o,
                      rra_dtype out_dtype, const int32_t* src_idx, int N, void* stream) {
  RRA_TRY(check_attend(qp, kp, vp, cu_seqlens, B, max_seqlen, H, d, scale, in_dtype, o, out_dtype, src_idx, N));
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  RRA_TRY(enqueue_attend(*st, qp, kp, vp, cu_seqlens, B, max_seqlen, H, scale, in_dtype, o, out_dtype,
                         src_idx, src_idx ? N : 0, static_cast<cudaStream_t>(stream)));
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_attend_wait(const void* qp, const void* kp, const void* vp, const int32_t* cu_seqlens, int B,
                           int max_seqlen, int H, int d, float scale, rra_dtype in_dtype, void* o,
                           rra_dtype out_dtype, const int32_t* src_idx, int N, void* stream) {
  RRA_TRY(check_attend(qp, kp, vp, cu_seqlens, B, max_seqlen, H, d, scale, in_dtype, o, out_dtype, src_idx, N));
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(s, &cap);
  if (ce != cudaSuccess) return cuda_fail(ce, "attend_wait: cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone)
    return fail(RRA_ERR_INVALID_ARG, "attend_wait blocks on its result and cannot be captured in a graph");
  std::lock_guard<std::mutex> lock(st->wait_mutex);
  RRA_TRY(done_signal_state(*st));
  if (++st->ticket == 0) st->ticket = 1;   // 0 is the word's initial value
  const uint32_t ticket = st->ticket;
  const DoneSignal sig{st->done_count, st->ctas_counted, st->host_count ? nullptr : st->host_word_dev, ticket};
  uint32_t ctas = 0;
  RRA_TRY(enqueue_attend(*st, qp, kp, vp, cu_seqlens, B, max_seqlen, H, scale, in_dtype, o, out_dtype, src_idx,
                         src_idx ? N : 0, s, &sig, &ctas));
  st->ctas_counted += ctas;   // every CTA of the launch will add one to the count
  g_launches += 1;
  const uint32_t want = st->host_count ? st->ctas_counted : ticket;
  // Poll the word for up to ~2 ms (a serving-size call lands in a few us);
  // a longer call is handed to a stream synchronisation, which also
  // surfaces an asynchronous error.
  const auto t0 = std::chrono::steady_clock::now();
  for (uint32_t spin = 1;; ++spin) {
    if (__atomic_load_n(st->host_word, __ATOMIC_ACQUIRE) == want) return RRA_OK;
    if ((spin & 1023u) == 0u && std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(2)) break;
  }
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "attend_wait: stream sync");
  if (__atomic_load_n(st->host_word, __ATOMIC_ACQUIRE) != want) {
    // Re-read the count so that later calls aim at the right total.
    uint32_t count = 0;
    if (st->host_count)
      st->ctas_counted = __atomic_load_n(st->host_word, __ATOMIC_ACQUIRE);
    else if (cudaMemcpy(&count, st->done_count, sizeof(count), cudaMemcpyDeviceToHost) == cudaSuccess)
      st->ctas_counted = count;
    return fail(RRA_ERR_CUDA, "attend_wait: the kernel finished without publishing its completion word");
  }
  return RRA_OK;
}

rra_status rra_attend_gather(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                             const int32_t* src_idx, int B, int N, int H, int d, float scale, rra_dtype in_dtype,
                             void* out, rra_dtype out_dtype, void* stream) {
  RRA_TRY(check_shape(B, N, H, d));
  if (!valid_in(in_dtype)) return fail(RRA_ERR_INVALID_ARG, "input dtype invalid");
  if (!valid_out(out_dtype)) return fail(RRA_ERR_INVALID_ARG, "output dtype invalid");
  if (!finite(scale)) return fail(RRA_ERR_INVALID_ARG, "scale is not finite");
  RRA_CHECK_PTR(q);
  RRA_CHECK_PTR(k);
  RRA_CHECK_PTR(v);
  RRA_CHECK_PTR(out);
  if (cu_seqlens == nullptr || src_idx == nullptr) return fail(RRA_ERR_INVALID_ARG, "index buffer is null");
  if (!attend_tc_available()) return fail(RRA_ERR_CUDA, "attend_gather: tensor-map encoder unavailable");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  AttendArgs a{};
  a.qp = q;
  a.kp = k;
  a.vp = v;
  a.cu_seqlens = cu_seqlens;
  a.src_idx = src_idx;
  a.o = out;
  a.B = B;
  a.H = H;
  a.N = N;
  a.max_seqlen = N;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = error_word(*st);
  a.wait_limit = g_wait_limit.load();
  cudaError_t e = launch_attend_tc_gather(a, in_dtype, out_dtype, st->num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attend (gather) launch");
  g_launches += 1;
  return RRA_OK;
}

// Checks of the class-token side output shared by rra_attend_cls and rra_attend_rows.
rra_status check_cls(const float* cls, int cls_stride, int max_seqlen, rra_dtype in_dtype, rra_dtype out_dtype) {
  if (cls == nullptr) return RRA_OK;
  if (!aligned16(cls)) return fail(RRA_ERR_MISALIGNED, "cls not 16-byte aligned");
  if (out_dtype != in_dtype) return fail(RRA_ERR_UNSUPPORTED, "a cls output needs out_dtype == in_dtype");
  const int need = (max_seqlen + 15) & ~15;
  if (cls_stride < need || cls_stride % 4 != 0)
    return fail(RRA_ERR_INVALID_ARG, "cls_stride=%d: a multiple of 4, at least %d", cls_stride, need);
  return RRA_OK;
}

rra_status rra_attend_cls(const void* qp, const void* kp, const void* vp, const int32_t* cu_seqlens, int B,
                          int max_seqlen, int H, int d, float scale, rra_dtype in_dtype, void* o, rra_dtype out_dtype,
                          float* cls, int cls_stride, void* stream) {
  RRA_TRY(check_attend(qp, kp, vp, cu_seqlens, B, max_seqlen, H, d, scale, in_dtype, o, out_dtype, nullptr, 0));
  if (cls == nullptr) return fail(RRA_ERR_INVALID_ARG, "cls is null");
  RRA_TRY(check_cls(cls, cls_stride, max_seqlen, in_dtype, out_dtype));
  if (static_cast<long long>(B) * H * cls_stride >= (1LL << 31)) return fail(RRA_ERR_UNSUPPORTED, "cls too large");
  if (!attend_tc_available()) return fail(RRA_ERR_CUDA, "attend_cls: tensor-map encoder unavailable");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  AttendArgs a{};
  a.qp = qp;
  a.kp = kp;
  a.vp = vp;
  a.cu_seqlens = cu_seqlens;
  a.o = o;
  a.B = B;
  a.H = H;
  a.N = max_seqlen;
  a.max_seqlen = max_seqlen;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = error_word(*st);
  a.wait_limit = g_wait_limit.load();
  a.cls = cls;
  a.cls_stride = cls_stride;
  cudaError_t e = launch_attend_tc(a, in_dtype, out_dtype, st->num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attend (cls) launch");
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_attend_rows(const void* q, const void* k, const void* v, long long src_rows, const int32_t* rows,
                           const int32_t* cu_seqlens, int B, int max_seqlen, int H, int d, float scale,
                           rra_dtype in_dtype, void* o, rra_dtype out_dtype, float* cls, int cls_stride,
                           void* stream) {
  RRA_TRY(check_attend(q, k, v, cu_seqlens, B, max_seqlen, H, d, scale, in_dtype, o, out_dtype, nullptr, 0));
  if (rows == nullptr) return fail(RRA_ERR_INVALID_ARG, "rows is null");
  if (src_rows < 1) return fail(RRA_ERR_INVALID_ARG, "src_rows=%lld < 1", src_rows);
  if (src_rows * H * d >= (1LL << 31)) return fail(RRA_ERR_UNSUPPORTED, "src_rows*H*d >= 2^31");
  RRA_TRY(check_cls(cls, cls_stride, max_seqlen, in_dtype, out_dtype));
  if (cls != nullptr && static_cast<long long>(B) * H * cls_stride >= (1LL << 31))
    return fail(RRA_ERR_UNSUPPORTED, "cls too large");
  if (!attend_tc_available()) return fail(RRA_ERR_CUDA, "attend_rows: tensor-map encoder unavailable");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  AttendArgs a{};
  a.cls = cls;
  a.cls_stride = cls_stride;
  a.qp = q;
  a.kp = k;
  a.vp = v;
  a.cu_seqlens = cu_seqlens;
  a.src_idx = rows;
  a.src_rows = src_rows;
  a.o = o;
  a.B = B;
  a.H = H;
  a.N = max_seqlen;
  a.max_seqlen = max_seqlen;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = error_word(*st);
  a.wait_limit = g_wait_limit.load();
  cudaError_t e = launch_attend_tc_rows(a, in_dtype, out_dtype, st->num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attend (rows) launch");
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_unpack(const void* op, const int32_t* dst_idx, int B, int N, int H, int d, rra_dtype dtype,
                      void* out, void* stream) {
  RRA_TRY(check_shape(B, N, H, d));
  if (!valid_out(dtype)) return fail(RRA_ERR_INVALID_ARG, "dtype invalid");
  RRA_CHECK_PTR(op);
  RRA_CHECK_PTR(out);
  if (dst_idx == nullptr) return fail(RRA_ERR_INVALID_ARG, "dst_idx is null");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  UnpackArgs a{};
  a.op = static_cast<const uint4*>(op);
  a.dst_idx = dst_idx;
  a.out = static_cast<uint4*>(out);
  a.B = B;
  a.N = N;
  a.row_vecs = H * d * dtype_bytes(dtype) / 16;
  a.err = error_word(*st);
  cudaError_t e = launch_unpack(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "unpack launch");
  g_launches += 1;
  return RRA_OK;
}

rra_status rra_pipeline(const uint8_t* keep, const void* q, const void* k, const void* v, int B, int N,
                        int H, int d, float scale, rra_dtype in_dtype, void* out, rra_dtype out_dtype,
                        void* workspace, size_t workspace_bytes, void* stream) {
  PipelineArgs p{keep, q, k, v, B, N, H, d, scale, in_dtype, out_dtype, out, workspace, workspace_bytes};
  RRA_TRY(check_pipeline(p));
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  RRA_TRY(enqueue_pipeline(*st, p, static_cast<cudaStream_t>(stream)));
  g_launches += pipeline_launches(*st, p);
  return RRA_OK;
}

rra_status rra_pipeline_host(const uint8_t* keep_h, const void* q_h, const void* k_h, const void* v_h,
                             int B, int N, int H, int d, float scale, rra_dtype in_dtype, void* out_h,
                             rra_dtype out_dtype, uint8_t* keep_d, void* q_d, void* k_d, void* v_d,
                             void* out_d, void* workspace, size_t workspace_bytes, void* stream) {
  PipelineArgs p{keep_d, q_d, k_d, v_d, B, N, H, d, scale, in_dtype, out_dtype, out_d, workspace,
                 workspace_bytes};
  RRA_TRY(check_pipeline(p));
  if (keep_h == nullptr || q_h == nullptr || k_h == nullptr || v_h == nullptr || out_h == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "host buffer is null");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t tokens = static_cast<size_t>(B) * N;
  const size_t in_bytes = tokens * H * d * dtype_bytes(in_dtype);
  const size_t out_bytes = tokens * H * d * dtype_bytes(out_dtype);
  cudaError_t e;
  if ((e = cudaMemcpyAsync(keep_d, keep_h, tokens, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "keep H2D");
  if ((e = cudaMemcpyAsync(q_d, q_h, in_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "q H2D");
  if ((e = cudaMemcpyAsync(k_d, k_h, in_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "k H2D");
  if ((e = cudaMemcpyAsync(v_d, v_h, in_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "v H2D");
  RRA_TRY(enqueue_pipeline(*st, p, s));
  g_launches += pipeline_launches(*st, p);
  if ((e = cudaMemcpyAsync(out_h, out_d, out_bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "out D2H");
  return RRA_OK;
}

rra_status rra_pipeline_mapped(const uint8_t* keep_h, const void* q_h, const void* k_h, const void* v_h,
                               int B, int N, int H, int d, float scale, rra_dtype in_dtype, void* out_h,
                               rra_dtype out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  const void* host[5] = {keep_h, q_h, k_h, v_h, out_h};
  const char* names[5] = {"keep_h", "q_h", "k_h", "v_h", "out_h"};
  void* mapped[5] = {};
  for (int i = 0; i < 5; ++i) {
    if (host[i] == nullptr) return fail(RRA_ERR_INVALID_ARG, "%s is null", names[i]);
    mapped[i] = mapped_host_ptr(host[i]);
    if (mapped[i] == nullptr)
      return fail(RRA_ERR_INVALID_ARG, "%s is not page-locked host memory the device can reach", names[i]);
  }
  PipelineArgs p{static_cast<const uint8_t*>(mapped[0]), mapped[1], mapped[2], mapped[3], B, N, H, d, scale,
                 in_dtype, out_dtype, mapped[4], workspace, workspace_bytes};
  RRA_TRY(check_pipeline(p));
  if (!is_device_memory(workspace)) return fail(RRA_ERR_INVALID_ARG, "workspace is not device memory");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long units = static_cast<long long>(B) * H * ((N + 127) / 128);
  if (pipeline_fused() && units <= st->num_sms) {
    // One launch: the tcgen05 kernel scans the mask, copies the kept rows
    // in with cp.async and writes every output row with plain stores.  Only
    // while each CTA has at most one (image, head, query tile) unit: larger
    // batches move more bytes than latency, and there pack's coalesced
    // 256-thread row copies use the link better than one loading warp per
    // CTA (measured on B=64: 142 against 190 us at 80% pruning, 399 against
    // 740 us dense).  The warp-specialised kernel even where the device
    // pipeline takes the small-grid one: its producer warp writes the
    // pruned rows as whole tokens right behind its first loads, and the
    // small-grid kernel's step took 9.8-10.4 against 9.1 us at serving B=4.
    AttendArgs a{};
    a.keep = p.keep;
    a.qp = p.q;
    a.kp = p.k;
    a.vp = p.v;
    a.o = p.out;
    a.B = p.B;
    a.H = p.H;
    a.N = p.N;
    a.max_seqlen = p.N;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.err = error_word(*st);
    a.wait_limit = g_wait_limit.load();
    cudaError_t e = launch_attend_tc_fused_host(a, p.in, p.out_dt, st->num_sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "mapped pipeline launch");
    g_launches += 1;
    return RRA_OK;
  }
  RRA_TRY(enqueue_packed_pipeline(*st, p, s, /*coalesced_out=*/true));
  g_launches += 2;
  return RRA_OK;
}

rra_status rra_plan_create(const uint8_t* keep, const void* q, const void* k, const void* v, int B, int N,
                           int H, int d, float scale, rra_dtype in_dtype, void* out, rra_dtype out_dtype,
                           void* workspace, size_t workspace_bytes, rra_plan** plan) {
  if (plan == nullptr) return fail(RRA_ERR_INVALID_ARG, "plan is null");
  *plan = nullptr;
  PipelineArgs p{keep, q, k, v, B, N, H, d, scale, in_dtype, out_dtype, out, workspace, workspace_bytes};
  RRA_TRY(check_pipeline(p));
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  // Run once eagerly on a private stream: loads the kernels' modules before
  // capture and surfaces launch errors with a plain status.
  cudaStream_t s = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreate");
  rra_status rs = enqueue_pipeline(*st, p, s);
  if (rs == RRA_OK) {
    g_launches += pipeline_launches(*st, p);
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) rs = cuda_fail(e, "plan warm-up");
  }
  cudaGraph_t graph = nullptr;
  if (rs == RRA_OK) {
    e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
      rs = cuda_fail(e, "cudaStreamBeginCapture");
    } else {
      rra_status cap = enqueue_pipeline(*st, p, s);
      e = cudaStreamEndCapture(s, &graph);
      if (cap != RRA_OK) rs = cap;
      else if (e != cudaSuccess) rs = cuda_fail(e, "cudaStreamEndCapture");
    }
  }
  cudaGraphExec_t exec = nullptr;
  if (rs == RRA_OK) {
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) rs = cuda_fail(e, "cudaGraphInstantiate");
  }
  cudaStreamDestroy(s);
  if (rs != RRA_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rs;
  }
  rra_plan* pl = new rra_plan;
  pl->graph = graph;
  pl->exec = exec;
  pl->launches = pipeline_launches(*st, p);
  *plan = pl;
  return RRA_OK;
}

rra_status rra_plan_launch(rra_plan* plan, void* stream) {
  if (plan == nullptr || plan->exec == nullptr) return fail(RRA_ERR_INVALID_ARG, "plan is null");
  cudaError_t e = cudaGraphLaunch(plan->exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
  g_launches += static_cast<uint64_t>(plan->launches);
  return RRA_OK;
}

void rra_plan_destroy(rra_plan* plan) {
  if (plan == nullptr) return;
  if (plan->exec) cudaGraphExecDestroy(plan->exec);
  if (plan->graph) cudaGraphDestroy(plan->graph);
  delete plan;
}

rra_status rra_get_device_error(int32_t* code, int clear) {
  if (code == nullptr) return fail(RRA_ERR_INVALID_ARG, "code is null");
  DeviceState* st = nullptr;
  RRA_TRY(device_state(&st));
  cudaError_t e = cudaMemcpy(code, st->err, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error");
  if (clear) {
    e = cudaMemset(st->err, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "clear device error");
  }
  return *code == 0 ? RRA_OK : RRA_ERR_DEVICE;
}

rra_status rra_bind_error_word(int32_t* word) {
  if (word != nullptr && (reinterpret_cast<uintptr_t>(word) & 3u) != 0)
    return fail(RRA_ERR_MISALIGNED, "error word not 4-byte aligned");
  g_bound_error_word = word;
  return RRA_OK;
}

rra_status rra_read_error_word(int32_t* word, int32_t* code, int clear) {
  if (word == nullptr || code == nullptr) return fail(RRA_ERR_INVALID_ARG, "word or code is null");
  cudaError_t e = cudaMemcpy(code, word, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (clear) {
    e = cudaMemset(word, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  }
  return *code == 0 ? RRA_OK : RRA_ERR_DEVICE;
}

long long rra_set_wait_limit(long long cycles) {
  if (cycles < 0) return -1;
  return g_wait_limit.exchange(cycles);
}

rra_status rra_time_attend_host(const void* qp, const void* kp, const void* vp, const int32_t* cu_seqlens,
                                int B, int max_seqlen, int H, int d, float scale, rra_dtype in_dtype,
                                void* o, rra_dtype out_dtype, const int32_t* src_idx, int N, void* stream,
                                int warmup, int reps, double* samples_us) {
  if (reps < 1 || warmup < 0 || samples_us == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "bad timing arguments");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < warmup + reps; ++i) {
    const auto t0 = std::chrono::steady_clock::now();
    rra_status rs = rra_attend(qp, kp, vp, cu_seqlens, B, max_seqlen, H, d, scale, in_dtype, o, out_dtype,
                               src_idx, N, stream);
    if (rs != RRA_OK) return rs;
    cudaError_t e = cudaStreamSynchronize(s);
    const auto t1 = std::chrono::steady_clock::now();
    if (e != cudaSuccess) return cuda_fail(e, "sync");
    if (i >= warmup) samples_us[i - warmup] = std::chrono::duration<double, std::micro>(t1 - t0).count();
  }
  return RRA_OK;
}

rra_status rra_time_attend_wait_host(const void* qp, const void* kp, const void* vp, const int32_t* cu_seqlens,
                                     int B, int max_seqlen, int H, int d, float scale, rra_dtype in_dtype,
                                     void* o, rra_dtype out_dtype, const int32_t* src_idx, int N, void* stream,
                                     int warmup, int reps, double* samples_us) {
  if (reps < 1 || warmup < 0 || samples_us == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "bad timing arguments");
  for (int i = 0; i < warmup + reps; ++i) {
    const auto t0 = std::chrono::steady_clock::now();
    rra_status rs = rra_attend_wait(qp, kp, vp, cu_seqlens, B, max_seqlen, H, d, scale, in_dtype, o, out_dtype,
                                    src_idx, N, stream);
    const auto t1 = std::chrono::steady_clock::now();
    if (rs != RRA_OK) return rs;
    if (i >= warmup) samples_us[i - warmup] = std::chrono::duration<double, std::micro>(t1 - t0).count();
  }
  return RRA_OK;
}

rra_status rra_time_plan_host(rra_plan* plan, void* stream, int warmup, int reps, double* samples_us) {
  if (reps < 1 || warmup < 0 || samples_us == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "bad timing arguments");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < warmup + reps; ++i) {
    const auto t0 = std::chrono::steady_clock::now();
    rra_status rs = rra_plan_launch(plan, stream);
    if (rs != RRA_OK) return rs;
    cudaError_t e = cudaStreamSynchronize(s);
    const auto t1 = std::chrono::steady_clock::now();
    if (e != cudaSuccess) return cuda_fail(e, "sync");
    if (i >= warmup) samples_us[i - warmup] = std::chrono::duration<double, std::micro>(t1 - t0).count();
  }
  return RRA_OK;
}

rra_status rra_time_null_host(void* stream, int warmup, int reps, double* samples_us) {
  if (reps < 1 || warmup < 0 || samples_us == nullptr)
    return fail(RRA_ERR_INVALID_ARG, "bad timing arguments");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < warmup + reps; ++i) {
    const auto t0 = std::chrono::steady_clock::now();
    null_kernel<<<1, 32, 0, s>>>();
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    const auto t1 = std::chrono::steady_clock::now();
    if (e != cudaSuccess) return cuda_fail(e, "null kernel");
    if (i >= warmup) samples_us[i - warmup] = std::chrono::duration<double, std::micro>(t1 - t0).count();
  }
  return RRA_OK;
}

}  // extern "C"

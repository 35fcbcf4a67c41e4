// Bidirectional ragged attention, sm_103a tensor-core kernel: TMA tile
// loads, tcgen05.mma with TMEM accumulators, warp-specialised.
//
// Follows "Dispatch-Aware Ragged Attention for Pruned Vision Transformers",
// abstract (non-causal attention over pruned ViT sequences of at most 197 /
// 577 tokens) and the agents-report.net article, method overview bullet 2
// (attention computed directly on the compact buffer).
//
// Work unit = (image b, head h, tile of 128 query rows).  Persistent CTAs of
// 192 threads walk the units with a grid stride; a unit whose tile starts
// past the image's length is skipped.  Per unit, keys stream in chunks of
// 64; an item is one (unit, key chunk).  Warp roles:
//
//   warp 4     loads: per item, TMA copies of the chunk's K and V rows into a
//              2-stage ring (and, on a unit's first item, of the Q tile),
//              128-byte swizzle: 32-row boxes of packed tensors, gather4 of
//              kept rows of padded tensors (3-D boxes where an image keeps
//              every token), or, for tensors in host memory, 16-byte cp.async
//              copies into the same layout.  In the fused pipeline this warp
//              also scans the image's keep row (kept positions -> a shared
//              list) and writes +0 to the output rows of pruned positions;
//   warp 5     tensor-core products, issued by one elected lane of the
//              converged warp: S = Q K^T (M=128, N=chunk rounded up to 16,
//              K=64) into TMEM columns 0..63, and O += P_hi V + P_lo V (M=128,
//              N=64, K=chunk) with P read from TMEM and O accumulating in
//              TMEM columns 64..127.  The next S product is issued the moment
//              this P.V product has finished reading P;
//   warps 0-3  softmax, thread r owning query row r (TMEM lane r): the row's
//              max over the chunk, exponentials in base 2 against a per-row
//              reference, P written over S as two bf16/fp16 parts; after a
//              unit's last item, the epilogue (normalise, store the row).
//
// The reference of a row is its max over the unit's first chunk; it moves
// (rescaling O in TMEM, which is stable then: the previous P.V product has
// finished before this S product was issued) only when a later chunk's max
// exceeds it by more than 8 in the log2 domain, so every weight is at most
// 2^8.  A one-token image's single weight is exactly 1, so such a row
// returns V bit for bit.  P is split because one bf16 rounding of the weights alone
// leaves up to ~2e-3 of output error at these lengths; hi + lo carries ~16
// bits.  Keys past the image's end are masked (p = 0), and the V rows the
// product reads past the end are either a repeated finite row (gathered
// loads) or zeroed in shared memory (packed loads), so whatever the buffer
// holds there (even NaN) never reaches a kept output.  Every mbarrier wait
// is bounded by a clock-cycle limit and gives up early once another warp
// has raised the CTA's abort flag; then the CTA records
// RRA_DEVERR_WAIT_TIMEOUT, waits (bounded) for its own copies and products
// to land, frees its TMEM and returns.
//
// Launches carry programmatic stream serialisation: a CTA's set-up overlaps
// the previous kernel's tail, a griddepcontrol.wait precedes every global
// access, and each CTA releases the next kernel's launch once it has issued
// all its work.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "softmax_tc.cuh"

namespace rra {
namespace {

constexpr int BM = 128;        // query rows per unit (= TMEM lanes)
constexpr int BN = 64;         // keys per chunk (= columns of the S buffer)
constexpr int CONSUMERS = 128;             // warps 0-3: softmax and epilogue
constexpr int PRODUCER_WARP = 4;           // TMA loads (+ mask scan, zero fill)
constexpr int MMA_WARP = 5;                // tcgen05.mma issue
constexpr int THREADS = CONSUMERS + 64;
constexpr int BOX = 32;        // rows per TMA box (packed inputs)
constexpr int CTAS_PER_SM = 4;
constexpr int STAGES = 2;      // K/V chunk ring

constexpr uint32_t Q_BYTES = BM * 128;                 // 128 rows x 128 B
constexpr uint32_t KV_BYTES = BN * 128;                //  64 rows x 128 B
constexpr uint32_t OFF_Q = 0;                          // one Q tile
constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;            // K[STAGES]
constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;  // V[STAGES]
constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
// mbarriers (8 B each) and words, as offsets from OFF_BAR.
constexpr uint32_t B_FULL = 0;        // [STAGES] item loaded (TMA bytes + producer arrive)
constexpr uint32_t B_EMPTY = 16;      // [STAGES] item's K/V consumed (its P.V product done)
constexpr uint32_t B_QEMPTY = 32;     // unit's last S product done: Q buffer free
constexpr uint32_t B_SFULL = 40;      // S product done
constexpr uint32_t B_SFREE = 48;      // P.V product done (S/P buffer free)
constexpr uint32_t B_PREADY = 56;     // P written (128 consumer arrivals)
constexpr uint32_t B_OFULL = 64;      // unit's last P.V product done
constexpr uint32_t B_OEMPTY = 72;     // unit's O read out (128 consumer arrivals)
constexpr uint32_t B_DRAIN = 80;      // every product issued has completed
constexpr uint32_t W_TMEM = 88;       // TMEM base written by tcgen05.alloc
constexpr uint32_t W_ABORT = 92;      // abort flag
constexpr uint32_t B_STAGED = 96;     // unit's output rows read back out of the stage (4 softmax warps)
// Item descriptors, one per stage, then (fused pipeline) POS_SLOTS lists of
// kept positions (int16, N each).
constexpr uint32_t DESC_BYTES = 48;
constexpr uint32_t OFF_DESC = OFF_BAR + 112;
// 1024 zero bytes: the source of the bulk copies that write the pruned rows
// (a token row of H = 12 heads takes two copies; each copy is one TMA
// operation, and halving their number from 512-byte copies cut 0.5 us from
// B=64 at 80-90% pruning; 1024 keeps four CTAs per SM at N = 577).
constexpr uint32_t ZERO_BYTES = 1024;
constexpr uint32_t OFF_ZERO = OFF_DESC + STAGES * DESC_BYTES;
constexpr uint32_t OFF_POS = OFF_ZERO + ZERO_BYTES;
// Five lists: the producer scans unit u + 5 only after the last S product
// of unit u + 3, which follows the P.V products of unit u + 2; by then every
// consumer has finished unit u's epilogue (the last reader of its list).
constexpr int POS_SLOTS = 5;
constexpr uint32_t SMEM_ALLOC = OFF_POS + 1024;        // + position lists; slack to align the base to 1024 B

// MODE_FUSED: the pruned rows are written by bulk copies (zero_pruned_tokens);
// MODE_FUSED_ROWS: by plain stores (zero_pruned_rows), for grids of at most
// one unit per SM, where the kernel is one latency chain per CTA;
// MODE_FUSED_HOST: MODE_FUSED_ROWS for keep/q/k/v/out in page-locked host
// memory: rows come in by 16-byte cp.async copies (completion counted on the
// stage's mbarrier) instead of TMA, and every output row leaves by plain stores.
enum { MODE_PACKED = 0, MODE_GATHER = 1, MODE_FUSED = 2, MODE_FUSED_ROWS = 3, MODE_FUSED_HOST = 4 };
constexpr uint32_t TMEM_COLS = 128;                    // S/P: cols [0,64); O: cols [64,128)
constexpr uint32_t TMEM_O = BN;

static_assert(OFF_POS % 16 == 0, "position lists must start 16-byte aligned");
static_assert(OFF_ZERO % 16 == 0, "bulk-copy source must be 16-byte aligned");
static_assert(ZERO_BYTES == 2 * 32 * 16, "the producer warp zeroes the buffer with two 16-byte stores per lane");
static_assert(OFF_DESC >= OFF_BAR + W_ABORT + 4, "descriptor ring overlaps the flags");

// Loads of one item for an image whose every token is kept (position t is
// token t): 32-row groups inside the image as one 3-D box each, the partial
// last group by gather4, repeating its last row.  Kept out of line so that
// the gather path's code is laid out as without it.
__device__ __noinline__ void issue_whole_loads(int lane, int qgroups, int kgroups, int row0, int h, int H, int q0,
                                                int rows_q, int k0, int n_c, uint32_t sq, uint32_t sk, uint32_t sv,
                                                uint32_t bar, const CUtensorMap* mq, const CUtensorMap* mk,
                                                const CUtensorMap* mv, const CUtensorMap* mq3,
                                                const CUtensorMap* mk3, const CUtensorMap* mv3) {
  if (lane < qgroups) {
    const int G = lane >> 3;
    if (32 * G + 32 <= rows_q) {
      if ((lane & 7) == 0) tma_load_3d(sq + G * 4096, mq3, 0, h, row0 + q0 + 32 * G, bar);
    } else {
      int rows[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) rows[i] = (row0 + min(q0 + 4 * lane + i, q0 + rows_q - 1)) * H + h;
      tma_gather4(sq + lane * 512, mq, rows, bar);
    }
  }
  const int g = lane & 15;
  if (g < kgroups) {
    const int G = g >> 3;
    if (32 * G + 32 <= n_c) {
      if ((g & 7) == 0) {
        if (lane < 16) tma_load_3d(sk + G * 4096, mk3, 0, h, row0 + k0 + 32 * G, bar);
        else tma_load_3d(sv + G * 4096, mv3, 0, h, row0 + k0 + 32 * G, bar);
      }
    } else {
      int rows[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) rows[i] = (row0 + min(k0 + 4 * g + i, k0 + n_c - 1)) * H + h;
      if (lane < 16) tma_gather4(sk + g * 512, mk, rows, bar);
      else tma_gather4(sv + g * 512, mv, rows, bar);
    }
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

// Whole output rows (all heads) of image b's pruned tokens -> +0, the share
// of the (b, h) unit: pruned tokens h, h + H, h + 2H, ... of the list the
// scan left at the end of `pos` (entries N-1, N-2, ...).  A token's row is
// H*64 contiguous outputs; each lane hands one row at a time to the TMA
// engine as bulk copies from the shared zero buffer, so the warp spends a
// few instructions per row and the writes proceed on their own.  Producer
// warp, 32 lanes; before the CTA exits it waits until the copies have read
// the zero buffer.
template <typename Tout>
__device__ __forceinline__ void zero_pruned_tokens(const AttendArgs& a, int b, int h, int npruned, uint32_t pos,
                                                   uint32_t zero, int lane) {
  const uint32_t row_bytes = static_cast<uint32_t>(a.H) * HD * static_cast<uint32_t>(sizeof(Tout));
  uint8_t* const img = static_cast<uint8_t*>(a.o) + static_cast<size_t>(b) * a.N * row_bytes;
  for (int r = h + lane * a.H; r < npruned; r += 32 * a.H) {
    const int j = ld_shared_u16(pos + 2u * static_cast<uint32_t>(a.N - 1 - r));
    uint8_t* row = img + static_cast<size_t>(j) * row_bytes;
    for (uint32_t off = 0; off < row_bytes; off += ZERO_BYTES)
      bulk_store(row + off, zero, row_bytes - off < ZERO_BYTES ? row_bytes - off : ZERO_BYTES);
  }
  bulk_commit();
}

// Whole output rows (all heads) of image b's pruned tokens -> +0 with plain
// stores, the share of the (b, h) unit: pruned tokens h, h + H, ... of the
// list at the back of `pos` (entries N-1, N-2, ...).  The warp writes each
// token's H*64 contiguous outputs with consecutive lanes on consecutive 16-byte
// vectors, so every store instruction covers whole 128-byte lines.  Used
// for an output in host memory: the positions come from the scan (the keep
// row is not read over the link again) and the writes cross the link as
// full lines.
template <typename Tout>
__device__ __forceinline__ void zero_listed_tokens(const AttendArgs& a, int b, int h, int npruned, uint32_t pos,
                                                   int lane) {
  const int vecs = a.H * HD * static_cast<int>(sizeof(Tout)) / 16;   // per token row
  uint4* img = reinterpret_cast<uint4*>(static_cast<Tout*>(a.o) + static_cast<size_t>(b) * a.N * a.H * HD);
  for (int r = h; r < npruned; r += a.H) {
    const size_t j = static_cast<size_t>(ld_shared_u16(pos + 2u * static_cast<uint32_t>(a.N - 1 - r)));
    uint4* row = img + j * vecs;
    for (int v = lane; v < vecs; v += 32) row[v] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Zero-fill schemes: per-head rows found by re-reading the keep row (plain
// stores), whole-token rows by bulk copies, whole-token rows from the scan's
// list of pruned positions (plain stores).
enum { ZF_MASK_ROWS = 0, ZF_BULK_TOKENS = 1, ZF_LIST_TOKENS = 2 };

// The (b, h) unit's part of the pruned-output zero fill, by scheme ZF.
template <typename Tout, int ZF>
__device__ __forceinline__ void zero_fill_share(const AttendArgs& a, int b, int h, int npruned, uint32_t pos,
                                                uint32_t zero, int lane) {
  if constexpr (ZF == ZF_BULK_TOKENS) zero_pruned_tokens<Tout>(a, b, h, npruned, pos, zero, lane);
  else if constexpr (ZF == ZF_LIST_TOKENS) zero_listed_tokens<Tout>(a, b, h, npruned, pos, lane);
  else zero_pruned_rows<Tout>(a, b, h, lane);
}

// Fused pipeline, called by the 32 lanes of the producer warp: the next unit
// at index >= u (stride `step`) whose query tile holds rows.  For every
// candidate the warp scans its image's keep row with ballots; the kept
// positions go, in order, to the front of the int16 list at shared address
// `pos` (N entries), the pruned ones to its back (entry N-1 first).  Each
// (image, head) pair's share of the pruned-token zero fill has exactly one
// owner: the image's first query tile with no rows, or, when every tile has
// rows, the last one.  A skipped candidate that owns the share does it here;
// for a returned owner the producer does it later, after the loads of the
// item that follows are in flight.  So every output row is written exactly
// once (images with no kept token too) and the zero fill stays off the path
// that feeds the tensor cores.  Giving the share to an empty tile rather
// than the first one moves it to the CTAs with the least real work (the
// grid stride hands the units with the highest indices, the later tiles,
// to the CTAs that got the fewest): measured on B=64 at 80% pruning, 10.8
// against 11.7 us.
template <typename Tout, int ZF>
__device__ Unit next_unit_fused(int u, int step, int units, int BH, const AttendArgs& a, int lane, uint32_t pos,
                                uint32_t zero) {
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
        const int kept_before = cnt + __popc(m & lt);
        if (flag[r]) {
          st_shared_u16(pos + 2u * static_cast<uint32_t>(kept_before), static_cast<uint32_t>(j));
        } else if (ZF != ZF_MASK_ROWS && j < a.N) {
          st_shared_u16(pos + 2u * static_cast<uint32_t>(a.N - 1 - (j - kept_before)), static_cast<uint32_t>(j));
        }
        cnt += __popc(m);
      }
    }
    const int q0 = qt * BM;
    if (q0 >= cnt) {
      if (q0 - BM < cnt) {   // the image's first empty query tile owns the share
        __syncwarp();
        zero_fill_share<Tout, ZF>(a, b, h, a.N - cnt, pos, zero, lane);
      }
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



// Source row of packed row t for the gather loads; a row outside [0, lim)
// records RRA_DEVERR_INDEX_RANGE and reads row 0 instead.
__device__ __forceinline__ int gather_row(const AttendArgs& a, int t, long long lim) {
  const int r = __ldg(a.src_idx + t);
  if (r < 0 || r >= lim) {
    record_error(a.err, RRA_DEVERR_INDEX_RANGE);
    return 0;
  }
  return r;
}

template <typename Tin, typename Tout, bool SCATTER, int MODE, bool LIMIT, bool CLS>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_q3,
                     const __grid_constant__ CUtensorMap tmap_k3, const __grid_constant__ CUtensorMap tmap_v3,
                     const AttendArgs a, int units, int pos_stride) {
  constexpr bool BF = IsBf16<Tin>::value == 1;
  constexpr bool GATHER = MODE != MODE_PACKED;
  constexpr bool FUSED = MODE == MODE_FUSED || MODE == MODE_FUSED_ROWS || MODE == MODE_FUSED_HOST;
  constexpr bool ZF_BULK = MODE == MODE_FUSED;
  constexpr int ZF = ZF_BULK ? ZF_BULK_TOKENS : (MODE == MODE_FUSED_HOST ? ZF_LIST_TOKENS : ZF_MASK_ROWS);
  constexpr bool HOSTLD = MODE == MODE_FUSED_HOST;   // cp.async loads (no tensor maps)
  // On packed or row-gathered inputs, 16-bit outputs of tiles with more than 64 rows leave
  // through the unit's last K/V stage (whole rows per store instruction);
  // smaller tiles (where the extra round trip through shared memory costs
  // more than it saves), fp32 outputs and the fused modes (whose producer
  // needs that stage back sooner) store row by row.
  constexpr bool STAGED = sizeof(Tout) == 2 && (MODE == MODE_PACKED || MODE == MODE_GATHER);
  constexpr int STAGE_MIN_ROWS = 65;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + OFF_Q;
  auto sK = [&](int i) { return base + OFF_K + i * KV_BYTES; };
  auto sV = [&](int i) { return base + OFF_V + i * KV_BYTES; };
  const uint32_t bars = base + OFF_BAR;
  auto bar_full = [&](int i) { return bars + B_FULL + 8 * i; };
  auto bar_empty = [&](int i) { return bars + B_EMPTY + 8 * i; };
  const uint32_t bar_qempty = bars + B_QEMPTY, bar_sfull = bars + B_SFULL, bar_sfree = bars + B_SFREE;
  const uint32_t bar_pready = bars + B_PREADY, bar_ofull = bars + B_OFULL, bar_oempty = bars + B_OEMPTY;
  const uint32_t bar_drain = bars + B_DRAIN, abort_flag = bars + W_ABORT;
  auto desc_addr = [&](int i) { return base + OFF_DESC + i * DESC_BYTES; };
  auto pos_addr = [&](int s) { return base + OFF_POS + s * pos_stride; };
  const volatile uint32_t* tmem_ptr = reinterpret_cast<const volatile uint32_t*>(gbase + OFF_BAR + W_TMEM);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    tmem_alloc(bars + W_TMEM, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int i = 0; i < STAGES; ++i) {
      // TMA: the producer's arrive + the copies' bytes; cp.async: one
      // arrival per producer lane when its copies land + lane 0's arrive.
      mbar_init(bar_full(i), HOSTLD ? 33 : 1);
      mbar_init(bar_empty(i), 1);
    }
    mbar_init(bar_qempty, 1);
    mbar_init(bar_sfull, 1);
    mbar_init(bar_sfree, 1);
    mbar_init(bar_pready, CONSUMERS);
    mbar_init(bar_ofull, 1);
    mbar_init(bar_oempty, CONSUMERS);
    mbar_init(bar_drain, 1);
    mbar_init(bars + B_STAGED, 4);
    st_shared_u32(abort_flag, 0u);
    fence_barrier_init();
  }
  const uint32_t zero_buf = base + OFF_ZERO;
  if (ZF_BULK && warp == PRODUCER_WARP) {
    st_shared_v4(zero_buf + 16 * lane, 0u, 0u, 0u, 0u);         // 2 x 32 lanes x 16 B = ZERO_BYTES
    st_shared_v4(zero_buf + 512 + 16 * lane, 0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  if (!HOSTLD && warp == PRODUCER_WARP && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  // Launched as a programmatic dependent of the kernel before it in the
  // stream: the set-up above (TMEM, barriers, descriptor prefetch) may run
  // while that kernel finishes; nothing in global memory is read or written
  // before its completion, which this waits for (at once if there is none).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int BH = a.B * a.H;
  const int step = gridDim.x;
  // The bound on one wait: a compile-time constant, except in the
  // instantiation for a launch made with a wait limit set (rra_set_wait_limit).
  const long long wlimit = LIMIT ? a.wait_limit : WAIT_LIMIT_CYCLES;
  // Rows the gather loads may read (row-gather inputs span a.src_rows rows).
  const long long src_lim = a.src_rows > 0 ? a.src_rows : static_cast<long long>(a.B) * a.N;
  bool bad = false;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ loads
    // Walks this CTA's items in order.  For each: waits until its stage
    // (and, on a unit's first item, the Q buffer) is free, publishes the
    // item's descriptor and issues the TMA loads that complete the stage's
    // full barrier.  Ends with a sentinel descriptor (plain arrive).
    uint32_t j = 0, uidx = 0;
    int zlast_b = -1, zlast_h = 0, zlast_n = 0;   // fused: the last unit's zero-fill share, if pending
    uint32_t zlast_pos = 0;
    Unit U;
    if constexpr (FUSED) U = next_unit_fused<Tout, ZF>(blockIdx.x, step, units, BH, a, lane, pos_addr(0), zero_buf);
    else U = next_unit(blockIdx.x, step, units, BH, a, lane == 0);
    bool done = false;
    while (!done && !bad) {
      const bool sentinel = U.u >= units;
      const int nch = sentinel ? 1 : U.nchunks;
      for (int c = 0; c < nch; ++c) {
        const int st = static_cast<int>(j % STAGES);
        if (j >= STAGES) bad |= !mbar_wait_or_abort(bar_empty(st), ((j / STAGES) - 1) & 1, abort_flag, wlimit);
        if (!sentinel && c == 0 && uidx >= 1) bad |= !mbar_wait_or_abort(bar_qempty, (uidx - 1) & 1, abort_flag, wlimit);
        bad = __any_sync(0xffffffffu, bad);
        if (bad) break;
        const uint32_t d = desc_addr(st);
        if (sentinel) {
          if (lane == 0) {
            st_shared_u32(d + 0, static_cast<uint32_t>(units));
            mbar_arrive(bar_full(st));
          }
          // This CTA has issued all its work: the next kernel in the stream
          // may start launching once every CTA got here.  (Triggered at the
          // start instead, the next grid's CTAs took the slots in the order
          // CTAs finished, which unbalanced the grid-stride unit sets:
          // +3 us on B=64 dense; here -0.8 us.)
          asm volatile("griddepcontrol.launch_dependents;" :::);
          if constexpr (HOSTLD) cp_async_arrive_noinc(bar_full(st));
          // The last unit's zero-fill share, after the end of work is
          // published: the other warps need not wait for it.
          if constexpr (FUSED) {
            if (zlast_b >= 0) zero_fill_share<Tout, ZF>(a, zlast_b, zlast_h, zlast_n, zlast_pos, zero_buf, lane);
          }
          done = true;
          break;
        }
        const int k0 = c * BN;
        const int n_c = min(BN, U.n - k0);
        if (lane == 0) {
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
        if constexpr (HOSTLD) {
          // 16-byte pieces, piece p = row p/8, chunk p%8, lanes striding
          // over them; rows past the tile's end repeat its last row (finite
          // V rows for the keys the products read past the image's end).
          const uint32_t pslot = pos_addr(static_cast<int>(uidx % POS_SLOTS));
          const size_t img = static_cast<size_t>(U.b) * a.N;
          const uint8_t* qg = static_cast<const uint8_t*>(a.qp);
          const uint8_t* kg = static_cast<const uint8_t*>(a.kp);
          const uint8_t* vg = static_cast<const uint8_t*>(a.vp);
          auto row_off = [&](int t) {
            return ((img + static_cast<size_t>(ld_shared_u16(pslot + 2 * t))) * a.H + U.h) * (HD * 2);
          };
          if (c == 0) {
            for (int p = lane; p < U.rows_q * 8; p += 32) {
              const int r = p >> 3, ch = p & 7;
              cp_async16(sQ + swz128(r, ch), qg + row_off(U.q0 + r) + ch * 16);
            }
          }
          const int nk = (n_c + 15) & ~15;
          for (int p = lane; p < nk * 8; p += 32) {
            const int r = p >> 3, ch = p & 7;
            const size_t off = row_off(k0 + min(r, n_c - 1)) + ch * 16;
            cp_async16(sK(st) + swz128(r, ch), kg + off);
            cp_async16(sV(st) + swz128(r, ch), vg + off);
          }
          cp_async_arrive_noinc(bar_full(st));
          if (lane == 0) mbar_arrive(bar_full(st));   // after the descriptor stores
        } else if constexpr (GATHER) {
          // K: lanes 0-15, V: lanes 16-31, one 4-row gather each; Q: up to 32 lanes.
          const int kgroups = ((n_c + 15) & ~15) / 4;
          const int qgroups = (c == 0) ? (U.rows_q + 3) / 4 : 0;
          if (lane == 0) mbar_expect_tx(bar_full(st), static_cast<uint32_t>((2 * kgroups + qgroups) * 512));
          __syncwarp();
          const uint32_t pslot = pos_addr(static_cast<int>(uidx % POS_SLOTS));
          bool whole = false;   // every token of the image kept: position t is token t
          if constexpr (FUSED) whole = U.n == a.N;
          if (whole) {
            issue_whole_loads(lane, qgroups, kgroups, U.b * a.N, U.h, a.H, U.q0, U.rows_q, k0, n_c, sQ, sK(st), sV(st),
                              bar_full(st), &tmap_q, &tmap_k, &tmap_v, &tmap_q3, &tmap_k3, &tmap_v3);
          } else {
            if (lane < qgroups) {
              int rows[4];
  #pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int t = min(U.q0 + 4 * lane + i, U.q0 + U.rows_q - 1);
                if constexpr (FUSED) rows[i] = (U.b * a.N + ld_shared_u16(pslot + 2 * t)) * a.H + U.h;
                else rows[i] = gather_row(a, U.s0 + t, src_lim) * a.H + U.h;
              }
              tma_gather4(sQ + lane * 512, &tmap_q, rows, bar_full(st));
            }
            const int g = lane & 15;
            if (g < kgroups) {
              int rows[4];
  #pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int t = min(k0 + 4 * g + i, k0 + n_c - 1);
                if constexpr (FUSED) rows[i] = (U.b * a.N + ld_shared_u16(pslot + 2 * t)) * a.H + U.h;
                else rows[i] = gather_row(a, U.s0 + t, src_lim) * a.H + U.h;
              }
              if (lane < 16) tma_gather4(sK(st) + g * 512, &tmap_k, rows, bar_full(st));
              else tma_gather4(sV(st) + g * 512, &tmap_v, rows, bar_full(st));
            }
          }
        } else if (lane == 0) {
          // 32-row boxes: up to two each for K and V, four for Q.
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
        if constexpr (HOSTLD) {
          // Output in host memory: an owning unit (the image's last query
          // tile, all tiles having rows) sends its share of the pruned rows
          // right behind its first loads, so the link carries the writes
          // while the unit computes.
          if (c == 0 && U.q0 == (units / BH - 1) * BM)
            zero_fill_share<Tout, ZF>(a, U.b, U.h, a.N - U.n, pos_addr(static_cast<int>(uidx % POS_SLOTS)), zero_buf,
                                      lane);
        }
        __syncwarp();
        ++j;
      }
      if (done || bad) break;
      const int zb = U.b, zh = U.h, zn = a.N - U.n, zq = U.q0;   // this unit's zero-fill share
      const uint32_t zpos = pos_addr(static_cast<int>(uidx % POS_SLOTS));
      ++uidx;
      if constexpr (FUSED)
        U = next_unit_fused<Tout, ZF>(U.u + step, step, units, BH, a, lane, pos_addr(uidx % POS_SLOTS), zero_buf);
      else U = next_unit(U.u + step, step, units, BH, a, lane == 0);
      if constexpr (FUSED) {
        // With the next unit scanned (and this unit's loads in flight), the
        // share of the image's pruned output rows if this unit owns it (the
        // last query tile, every tile having rows); after the last unit it
        // waits until the end of work is published.
        if (!HOSTLD && zq == (units / BH - 1) * BM) {
          if (U.u < units) {
            zero_fill_share<Tout, ZF>(a, zb, zh, zn, zpos, zero_buf, lane);
          } else {
            zlast_b = zb;
            zlast_h = zh;
            zlast_n = zn;
            zlast_pos = zpos;
          }
        }
      }
    }
    if constexpr (ZF_BULK) bulk_wait_read();   // the zero buffer must outlive the copies that read it
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ products
    // Per item j: S(j) (once its loads have landed; P.V(j-1) has finished
    // with the S/P columns, see the end of the loop); then, once the
    // consumers have written P(j), O += P(j) V (a unit's first one also
    // waits until the consumers have read out the previous unit's O); then
    // the wait for that product before S(j+1).  A unit's last S product
    // frees the Q buffer for the next unit's loads.
    const uint32_t tS = tmem, tO = tmem + TMEM_O;
    const uint32_t idesc_pv = idesc_f16(BF ? 1u : 0u, 1, BM, HD);
    uint32_t j = 0, ph_pready = 0, ph_sfree = 0, ustarted = 0;
    int nk16 = 0, c = 0, nch = 0;
    auto issue_s = [&](int st) {
      tc_fence_after();
      const uint32_t idesc_s = idesc_f16(BF ? 1u : 0u, 0, BM, nk16);
      const bool leader = elect_one();
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint64_t da = sdesc(sQ + kk * 32, 16, 1024), db = sdesc(sK(st) + kk * 32, 16, 1024);
        if (leader) umma_f16(tS, da, db, idesc_s, kk > 0 ? 1u : 0u);
      }
      if (leader) umma_commit(bar_sfull);
    };
    for (;; ++j) {
      // S(j): loads, descriptor, then the product.
      const int st = static_cast<int>(j % STAGES);
      bad |= !mbar_wait_or_abort(bar_full(st), (j / STAGES) & 1, abort_flag, wlimit);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      const uint32_t d = desc_addr(st);
      if (static_cast<int>(ld_shared_u32(d + 0)) >= units) break;   // sentinel
      const int n = static_cast<int>(ld_shared_u32(d + 12));
      const bool staged = STAGED && static_cast<int>(ld_shared_u32(d + 20)) >= STAGE_MIN_ROWS;
      nch = static_cast<int>(ld_shared_u32(d + 24));
      c = static_cast<int>(ld_shared_u32(d + 28));
      const int n_c = min(BN, n - c * BN);
      nk16 = (n_c + 15) & ~15;
      const bool first = c == 0, last = c == nch - 1;
      if constexpr (HOSTLD) fence_proxy_async();   // cp.async wrote the tiles through the generic proxy
      if constexpr (!GATHER) {
        // Packed boxes: V rows [n_c, nk16) enter the P.V product with p = 0;
        // make them finite zeros (the gathered path repeats a valid row).
        const int zvec = (nk16 - n_c) * 8;
        for (int zi = lane; zi < zvec; zi += 32)
          st_shared_v4(sV(st) + (n_c + (zi >> 3)) * 128 + (zi & 7) * 16, 0u, 0u, 0u, 0u);
        fence_proxy_async();
        __syncwarp();
      }
      issue_s(st);
      if (last && elect_one()) umma_commit(bar_qempty);

      // P(j) written, then the P.V product.
      bad |= !mbar_wait_or_abort(bar_pready, ph_pready, abort_flag, wlimit);
      ph_pready ^= 1;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      if (first && ustarted >= 1) {
        bad |= !mbar_wait_or_abort(bar_oempty, (ustarted - 1) & 1, abort_flag, wlimit);
        bad = __any_sync(0xffffffffu, bad);
        if (bad) break;
      }
      if (first) ++ustarted;
      tc_fence_after();
      {
        const bool leader = elect_one();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          if (kk * 16 < nk16) {
            const uint64_t db = sdesc(sV(st) + kk * 2048, KV_BYTES, 1024);
            if (leader) umma_f16_tmem_a(tO, tS + kk * 16, db, idesc_pv, (kk > 0 || !first) ? 1u : 0u);
          }
        }
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          if (kk * 16 < nk16) {
            const uint64_t db = sdesc(sV(st) + kk * 2048, KV_BYTES, 1024);
            if (leader) umma_f16_tmem_a(tO, tS + kk * 16 + 8, db, idesc_pv, 1u);
          }
        }
        // (A unit's last stage is handed back by the epilogue, which stages
        // 16-bit output rows in it.)
        if (leader && !(staged && last)) umma_commit(bar_empty(st));
        if (leader && last) umma_commit(bar_ofull);
        if (leader) umma_commit(bar_sfree);
      }
      bad |= !mbar_wait_or_abort(bar_sfree, ph_sfree, abort_flag, wlimit);
      ph_sfree ^= 1;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
    }
    if (!bad) {
      // Every product issued has completed (and with it the arrivals above).
      if (elect_one()) umma_commit(bar_drain);
      bad |= !mbar_wait_or_abort(bar_drain, 0, abort_flag, wlimit);
      bad = __any_sync(0xffffffffu, bad);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS_row = tmem + lane_off, tO_row = tmem + TMEM_O + lane_off;
    const float c2 = a.scale_log2;
    uint32_t uidx = 0, ph_sfull = 0;
    float m_run = 0.f, l_run = 0.f;   // this row's reference (log2 units) and weight sum
    long long out_elem = -1;          // this row's output offset in the current unit
    float* cls_row = nullptr;         // CLS: the unit's class-token row of a.cls (warp 0, first tile), or null
    // CLS: the class token's raw scores of the unit so far (lane 0 of warp 0
    // writes them chunk by chunk; the warp turns them into weights at the end).
    float* const cls_buf = reinterpret_cast<float*>(gbase + OFF_POS);
    for (uint32_t j = 0;; ++j) {
      const int st = static_cast<int>(j % STAGES);
      bad |= !mbar_wait_or_abort(bar_full(st), (j / STAGES) & 1, abort_flag, wlimit);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      const uint32_t d = desc_addr(st);
      if (static_cast<int>(ld_shared_u32(d + 0)) >= units) break;   // sentinel
      const int n = static_cast<int>(ld_shared_u32(d + 12));
      const int rows_q = static_cast<int>(ld_shared_u32(d + 20));
      const int nchunks = static_cast<int>(ld_shared_u32(d + 24));
      const int c = static_cast<int>(ld_shared_u32(d + 28));
      const int n_c = min(BN, n - c * BN);
      const int nk16 = (n_c + 15) & ~15;
      const bool rows_here = warp * 32 < rows_q;   // warp-uniform
      const bool last = (c == nchunks - 1);
      if (c == 0) {
        // Where this thread's row goes (element offset of its output row), or -1.
        const int h = static_cast<int>(ld_shared_u32(d + 4));
        const int s0 = static_cast<int>(ld_shared_u32(d + 8));
        const int q0 = static_cast<int>(ld_shared_u32(d + 16));
        const int i = q0 + tid;
        long long dst_row = -1;
        if (i < n) {
          dst_row = static_cast<long long>(s0) + i;
          if constexpr (FUSED) {
            const int ib = static_cast<int>(ld_shared_u32(d + 32));
            const int pslot = static_cast<int>(ld_shared_u32(d + 36));
            dst_row = static_cast<long long>(ib) * a.N + ld_shared_u16(pos_addr(pslot) + 2 * i);
          } else if constexpr (SCATTER) {
            dst_row = __ldg(a.src_idx + dst_row);
            if (dst_row < 0 || dst_row >= static_cast<long long>(a.B) * a.N) {
              record_error(a.err, RRA_DEVERR_INDEX_RANGE);
              dst_row = -1;
            }
          }
        }
        out_elem = dst_row < 0 ? -1 : (dst_row * a.H + h) * HD;
        if constexpr (CLS) {
          cls_row = nullptr;
          if (warp == 0 && q0 == 0) {
            const int ib = static_cast<int>(ld_shared_u32(d + 32));
            cls_row = a.cls + (static_cast<size_t>(ib) * a.H + h) * a.cls_stride;
          }
        }
      }
      bad |= !mbar_wait_or_abort(bar_sfull, ph_sfull, abort_flag, wlimit);
      ph_sfull ^= 1;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      tc_fence_after();

      if constexpr (CLS) {
        if (rows_here)
          softmax_chunk64<BF, true>(tS_row, tO_row, nk16, n_c, c, tid < rows_q, c2, m_run, l_run,
                                    (cls_row != nullptr && lane == 0) ? cls_buf + c * BN : nullptr);
      } else {
        if (rows_here) softmax_chunk64<BF>(tS_row, tO_row, nk16, n_c, c, tid < rows_q, c2, m_run, l_run);
      }
      tc_fence_before();
      mbar_arrive(bar_pready);
      if constexpr (CLS) {
        if (last && cls_row != nullptr) {
          // The class token's row is complete: its raw scores (stashed in
          // shared memory by lane 0) leave as weights 2^(c2*s - m) / l.
          const float m0 = __shfl_sync(0xffffffffu, m_run, 0);
          const float inv = 1.f / __shfl_sync(0xffffffffu, l_run, 0);
          __syncwarp();
          for (int i = lane; i < n; i += 32) cls_row[i] = fast_exp2(fmaf(cls_buf[i], c2, -m0)) * inv;
          __syncwarp();   // read out before lane 0 writes the next unit's scores
        }
      }

      if (last) {
        // Epilogue: this thread's row, normalised, to the packed or padded output.
        bad |= !mbar_wait_or_abort(bar_ofull, uidx & 1, abort_flag, wlimit);
        bad = __any_sync(0xffffffffu, bad);
        if (bad) break;
        tc_fence_after();
        if (STAGED && rows_q >= STAGE_MIN_ROWS) {
          // Each warp writes its 32 rows (128 bytes each) into 4 KB of the
          // unit's last K/V stage (swizzled by row), then stores them back
          // out with 8 lanes per row: every store instruction covers four
          // whole rows.  The stage goes back to the producer afterwards.
          const uint32_t stg = (warp < 2 ? sK(st) : sV(st)) + static_cast<uint32_t>(warp & 1) * 4096u;
          if (rows_here) {
            const float inv = 1.f / l_run;
#pragma unroll
            for (int g = 0; g < HD / 16; ++g) {
              float o[16];
              tmem_ld16(tO_row + g * 16, o);
              if (g == HD / 16 - 1) {
                tc_fence_before();
                mbar_arrive(bar_oempty);   // O is in registers: the next unit may overwrite it
              }
              uint32_t w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w[i] = pack2<Tout2<Tout>>(o[2 * i] * inv, o[2 * i + 1] * inv);
              st_shared_v4(stg + lane * 128 + (((2 * g) ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
              st_shared_v4(stg + lane * 128 + (((2 * g + 1) ^ (lane & 7)) << 4), w[4], w[5], w[6], w[7]);
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = 4 * i + (lane >> 3), cc = lane & 7;
              const long long dst = __shfl_sync(0xffffffffu, out_elem, rr);
              const uint4 v = ld_shared_v4(stg + rr * 128 + ((cc ^ (rr & 7)) << 4));
              if (dst >= 0) *reinterpret_cast<uint4*>(static_cast<Tout*>(a.o) + dst + cc * 8) = v;
            }
          } else {
            tc_fence_before();
            mbar_arrive(bar_oempty);
          }
          fence_proxy_async();   // these shared-memory accesses before the producer's next copies into the stage
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + B_STAGED);
          if (warp == 0) {
            bad |= !mbar_wait_or_abort(bars + B_STAGED, uidx & 1, abort_flag, wlimit);
            bad = __any_sync(0xffffffffu, bad);
            if (lane == 0 && !bad) mbar_arrive(bar_empty(st));
            if (bad) break;
          }
        } else {
          if (rows_here) {
            const float inv = 1.f / l_run;
            Tout* out = static_cast<Tout*>(a.o) + (out_elem < 0 ? 0 : out_elem);
#pragma unroll
            for (int g = 0; g < HD / 16; ++g) {
              float o[16];
              tmem_ld16(tO_row + g * 16, o);
              if (g == HD / 16 - 1) {
                tc_fence_before();
                mbar_arrive(bar_oempty);   // O is in registers: the next unit may overwrite it
              }
              if (out_elem >= 0) store16<Tout>(out + g * 16, o, inv);
            }
          } else {
            tc_fence_before();
            mbar_arrive(bar_oempty);
          }
        }
        ++uidx;
      }
    }
  }
  if (bad && lane == 0) {
    st_shared_u32(abort_flag, 1u);
    record_error(a.err, RRA_DEVERR_WAIT_TIMEOUT);
  }
  // Host completion word (rra_attend_wait): the packed and gather modes
  // write their output with plain stores only, all issued by now, so the
  // host may see the count move before the teardown below.
  if constexpr (!FUSED) {
    if (a.done_count != nullptr) signal_done(a);
  }

  // Teardown.  After an abort, copies or products still in flight get a
  // bounded grace period (~1 ms) to land before the TMEM is released and the
  // CTA exits.
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    if (lane == 0 && ld_shared_volatile_u32(abort_flag) != 0u) {
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    __syncwarp();
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

template <typename Tin, typename Tout, bool SCATTER, int MODE, bool LIMIT, bool CLS>
cudaError_t launch_tc_typed(const AttendArgs& a, int num_sms, cudaStream_t stream, uint32_t* ctas) {
  // Largest dynamic shared memory any launch of this instantiation asks for
  // (position lists for N <= 1024 in the fused mode).
  constexpr bool kFused = MODE == MODE_FUSED || MODE == MODE_FUSED_ROWS || MODE == MODE_FUSED_HOST;
  constexpr uint32_t kMaxSmem = SMEM_ALLOC + (kFused ? POS_SLOTS * 2048u : 0u) + (CLS ? 4096u : 0u);
  auto kernel = attend_tc_kernel<Tin, Tout, SCATTER, MODE, LIMIT, CLS>;
  static bool attr_set[kMaxDev] = {};
  static uint32_t occ_smem[kMaxDev] = {};
  static int occ_blocks[kMaxDev] = {};
  static std::mutex m;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  const int pos_stride = kFused ? ((2 * a.N + 15) & ~15) : 0;
  // CLS: the class-token score buffer (max_seqlen rounded up to 16 floats) where the position lists would be.
  const uint32_t cls_bytes = CLS ? static_cast<uint32_t>(((a.max_seqlen + 15) & ~15) * 4) : 0u;
  const uint32_t smem = SMEM_ALLOC + static_cast<uint32_t>(POS_SLOTS * pos_stride) + cls_bytes;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(m);
    if (!attr_set[dev]) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxSmem));
      if (e != cudaSuccess) return e;
      // All of the SM's unified L1/shared array as shared memory: four CTAs
      // of ~52 KB must be resident together.
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
    if (occ_smem[dev] != smem) {
      // Resident CTAs per SM at this shared-memory size (4 unless the
      // position lists of a long N push it lower); sizes the persistent grid.
      int per_sm_smem = 0, reserved = 0;
      e = cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
      if (e != cudaSuccess) return e;
      const int nb = per_sm_smem / (static_cast<int>(smem) + reserved);
      if (nb < 1) return cudaErrorInvalidConfiguration;
      occ_blocks[dev] = nb < CTAS_PER_SM ? nb : CTAS_PER_SM;
      occ_smem[dev] = smem;
    }
    per_sm = occ_blocks[dev];
  }
  const bool bf16 = IsBf16<Tin>::value == 1;
  CUtensorMap mq{}, mk{}, mv{}, mq3{}, mk3{}, mv3{};
  if constexpr (MODE == MODE_FUSED_HOST) {
    // cp.async loads: the kernel takes no tensor map (the zeroed ones are unused).
  } else if constexpr (MODE != MODE_PACKED) {
    const long long rows = (a.src_rows > 0 ? a.src_rows : static_cast<long long>(a.B) * a.N) * a.H;
    if ((e = make_gather_map(&mq, a.qp, rows, bf16)) != cudaSuccess) return e;
    if ((e = make_gather_map(&mk, a.kp, rows, bf16)) != cudaSuccess) return e;
    if ((e = make_gather_map(&mv, a.vp, rows, bf16)) != cudaSuccess) return e;
    if constexpr (kFused) {
      // 32-token boxes for images whose every token is kept
      const long long tokens = static_cast<long long>(a.B) * a.N;
      if ((e = make_map(&mq3, a.qp, a.H, tokens, bf16)) != cudaSuccess) return e;
      if ((e = make_map(&mk3, a.kp, a.H, tokens, bf16)) != cudaSuccess) return e;
      if ((e = make_map(&mv3, a.vp, a.H, tokens, bf16)) != cudaSuccess) return e;
    }
  } else {
    const long long rows = static_cast<long long>(a.B) * a.max_seqlen;
    if ((e = make_map(&mq, a.qp, a.H, rows, bf16)) != cudaSuccess) return e;
    if ((e = make_map(&mk, a.kp, a.H, rows, bf16)) != cudaSuccess) return e;
    if ((e = make_map(&mv, a.vp, a.H, rows, bf16)) != cudaSuccess) return e;
  }
  const int qtiles = (a.max_seqlen + BM - 1) / BM;
  const long long units = static_cast<long long>(a.B) * a.H * qtiles;
  const long long cap = static_cast<long long>(per_sm) * (num_sms > 0 ? num_sms : 152);
  const int grid = static_cast<int>(units < cap ? units : cap);
  AttendArgs b = a;
  if (b.done_count != nullptr) b.done_target += static_cast<uint32_t>(grid);
  if (ctas != nullptr) *ctas = static_cast<uint32_t>(grid);
  // Programmatic stream serialisation: the launch (and the kernel's set-up)
  // overlaps the tail of the previous kernel in the stream; the kernel waits
  // for that kernel's completion before touching global memory.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mq3, mk3, mv3, b, static_cast<int>(units), pos_stride);
}

// A launch made with a wait limit set runs its own instantiation, so that the
// kernels every other launch runs keep the bound a compile-time constant.
template <typename Tin, typename Tout, bool SCATTER, int MODE, bool CLS = false>
cudaError_t launch_tc_lim(const AttendArgs& a, int num_sms, cudaStream_t stream, uint32_t* ctas) {
  if (a.wait_limit > 0) return launch_tc_typed<Tin, Tout, SCATTER, MODE, true, CLS>(a, num_sms, stream, ctas);
  return launch_tc_typed<Tin, Tout, SCATTER, MODE, false, CLS>(a, num_sms, stream, ctas);
}

template <typename Tin, typename Tout>
cudaError_t launch_tc_out(const AttendArgs& a, int mode, int num_sms, cudaStream_t stream, uint32_t* ctas) {
  if (a.cls != nullptr) {
    // The class-token side output: packed outputs of the input's own type.
    if constexpr (std::is_same<Tin, Tout>::value) {
      if (mode == MODE_PACKED && a.src_idx == nullptr)
        return launch_tc_lim<Tin, Tout, false, MODE_PACKED, true>(a, num_sms, stream, ctas);
      if (mode == MODE_GATHER && a.src_rows > 0)
        return launch_tc_lim<Tin, Tout, false, MODE_GATHER, true>(a, num_sms, stream, ctas);
    }
    return cudaErrorInvalidValue;
  }
  if (mode == MODE_FUSED) {
    // Zero fill by bulk copies unless the grid has at most one unit per SM
    // (there the kernel is one latency chain per CTA and plain stores finish
    // sooner: measured 6.0 against 6.6 us on the serving workload).
    const long long units = static_cast<long long>(a.B) * a.H * ((a.max_seqlen + BM - 1) / BM);
    if (units <= (num_sms > 0 ? num_sms : 152))
      return launch_tc_lim<Tin, Tout, true, MODE_FUSED_ROWS>(a, num_sms, stream, ctas);
    return launch_tc_lim<Tin, Tout, true, MODE_FUSED>(a, num_sms, stream, ctas);
  }
  if (mode == MODE_FUSED_HOST) return launch_tc_lim<Tin, Tout, true, MODE_FUSED_HOST>(a, num_sms, stream, ctas);
  if (mode == MODE_GATHER) {
    if (a.src_rows > 0) return launch_tc_lim<Tin, Tout, false, MODE_GATHER>(a, num_sms, stream, ctas);
    return launch_tc_lim<Tin, Tout, true, MODE_GATHER>(a, num_sms, stream, ctas);
  }
  if (a.src_idx != nullptr) return launch_tc_lim<Tin, Tout, true, MODE_PACKED>(a, num_sms, stream, ctas);
  return launch_tc_lim<Tin, Tout, false, MODE_PACKED>(a, num_sms, stream, ctas);
}

template <typename Tin>
cudaError_t launch_tc_in(const AttendArgs& a, rra_dtype out, int mode, int num_sms, cudaStream_t stream,
                         uint32_t* ctas = nullptr) {
  if (out == RRA_BF16) return launch_tc_out<Tin, __nv_bfloat16>(a, mode, num_sms, stream, ctas);
  if (out == RRA_F16) return launch_tc_out<Tin, __half>(a, mode, num_sms, stream, ctas);
  return launch_tc_out<Tin, float>(a, mode, num_sms, stream, ctas);
}

}  // namespace

bool attend_tc_available() { return encode_fn(); }

cudaError_t launch_attend_tc(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms, cudaStream_t stream,
                             uint32_t* ctas) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (static_cast<long long>(a.B) * a.max_seqlen >= (1LL << 31)) return cudaErrorInvalidValue;
  if (in == RRA_BF16) return launch_tc_in<__nv_bfloat16>(a, out, MODE_PACKED, num_sms, stream, ctas);
  return launch_tc_in<__half>(a, out, MODE_PACKED, num_sms, stream, ctas);
}

cudaError_t launch_attend_tc_gather(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                    cudaStream_t stream) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (a.src_idx == nullptr) return cudaErrorInvalidValue;
  if (in == RRA_BF16) return launch_tc_in<__nv_bfloat16>(a, out, MODE_GATHER, num_sms, stream);
  return launch_tc_in<__half>(a, out, MODE_GATHER, num_sms, stream);
}

cudaError_t launch_attend_tc_rows(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                  cudaStream_t stream) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (a.src_idx == nullptr || a.src_rows < 1 || a.src_rows * a.H >= (1LL << 31)) return cudaErrorInvalidValue;
  if (static_cast<long long>(a.B) * a.max_seqlen >= (1LL << 31)) return cudaErrorInvalidValue;
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

cudaError_t launch_attend_tc_fused_host(const AttendArgs& a, rra_dtype in, rra_dtype out, int num_sms,
                                        cudaStream_t stream) {
  if (a.keep == nullptr || a.N > 1024) return cudaErrorInvalidValue;
  if (in == RRA_BF16) return launch_tc_in<__nv_bfloat16>(a, out, MODE_FUSED_HOST, num_sms, stream);
  return launch_tc_in<__half>(a, out, MODE_FUSED_HOST, num_sms, stream);
}

}  // namespace rra

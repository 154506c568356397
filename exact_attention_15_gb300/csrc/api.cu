// Host side of the C ABI declared in include/attn.h: argument validation,
// tensor-memory-accelerator descriptors, launch plans and the device error word.
// Order of work in every entry point: check arguments -> fill the parameter
// block -> launch (the order the FlashAttention-1 code layout describes for its
// C++ API: FlashAttention notes, xwysyy.cn, "code structure").
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/attn.h"
#include "attn_common.cuh"

namespace attn {
cudaError_t launch_attn_fwd(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p,
                            dim3 grid, cudaStream_t stream);
cudaError_t launch_attn_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tk_half,
                                 const CUtensorMap& tv, const FwdParams& p, dim3 grid,
                                 cudaStream_t stream);
cudaError_t launch_fwd_plan(const int* cu_seqlens, int B, int T, int H_q, int pair_heads,
                            int* seq_order, int* tile_start, int* tile_ctr, int* err,
                            cudaStream_t stream);
cudaError_t launch_seq_plan(const int* cu_seqlens, int B, int T, int rows, int units,
                            int* seq_order, int* tile_start, int* tile_ctr, int* err, int prof_id,
                            cudaStream_t stream);
cudaError_t launch_exp2_probe(const float* x, float* y, int n, int mode, cudaStream_t stream);
cudaError_t launch_stall_probe(int* err, long long limit, cudaStream_t stream);
int read_rescale_stats(unsigned long long* out, int reset);
cudaError_t launch_attn_bwd(const BwdParams& p, const CUtensorMap* maps, cudaStream_t stream,
                            long long rows_q, int n_sem, int n_work);
}  // namespace attn

using namespace attn;

// One error word per device (each device gets its own copy of this variable).
static __device__ int g_attn_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_dev_ok[kMaxDevices] = {};  // 0 unknown, 1 ok, -1 unsupported
// read by every launch without the lock, written under it
std::atomic<long long> g_wait_limit{2000000000ll};  // about one second of SM clock
std::atomic<int> g_fault{0};                        // host-injected fault, see attn_debug_inject
int g_bwd_variant = ATTN_BWD_ONE_CTA;   // backward main kernel at d = 128
int g_fwd_variant = ATTN_FWD_ONE_CTA;   // forward kernel at d_qk = d_v = 128
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return ATTN_ERR_NO_DEVICE;
  if (*dev < 0 || *dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
  return ATTN_OK;
}

// Per-device set-up: capability check and the address of the error word.
int device_setup(int dev, int** err_out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) {
      g_dev_ok[dev] = -1;
    } else {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_attn_error_word) != cudaSuccess) return ATTN_ERR_CUDA;
      g_err_ptr[dev] = static_cast<int*>(ptr);
      g_dev_ok[dev] = 1;
    }
  }
  if (g_dev_ok[dev] < 0) return ATTN_ERR_UNSUPPORTED_DEVICE;
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *err_out = g_err_ptr[dev];
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int g_sm_count[kMaxDevices] = {};

int sm_count(int dev) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

// Work-list metadata of the forward for packed sequences, one buffer per
// (device, stream): the sequence order, the first work tile of each sequence
// and the claim counter of the forward's schedule, written by the plan kernel
// right before the forward that reads them. Launches on one stream run in order, so they can share it; launches on
// different streams get different buffers. Buffers live until the process exits.
struct PlanBuf {
  int dev;
  cudaStream_t stream;
  int* ptr;
  int cap;  // sequences the arrays hold
};
std::mutex g_plan_mu;
std::vector<PlanBuf> g_plan;

int plan_buffer(int dev, cudaStream_t stream, int seqs, PlanBuf* out) {
  std::lock_guard<std::mutex> lock(g_plan_mu);
  PlanBuf* found = nullptr;
  for (PlanBuf& b : g_plan)
    if (b.dev == dev && b.stream == stream) found = &b;
  if (found && found->cap >= seqs) {
    *out = *found;
    return ATTN_OK;
  }
  const int cap = seqs > 1024 ? seqs : 1024;
  const size_t bytes = (2 * static_cast<size_t>(cap) + 2) * sizeof(int);
  if (found) {
    // growing: earlier launches on this stream may still read the old buffer
    if (cudaStreamSynchronize(stream) != cudaSuccess || cudaFree(found->ptr) != cudaSuccess)
      return ATTN_ERR_CUDA;
    found->ptr = nullptr;
  }
  void* ptr = nullptr;
  if (cudaMalloc(&ptr, bytes) != cudaSuccess) return ATTN_ERR_CUDA;
  if (found) {
    found->ptr = static_cast<int*>(ptr);
    found->cap = cap;
    *out = *found;
  } else {
    g_plan.push_back(PlanBuf{dev, stream, static_cast<int*>(ptr), cap});
    *out = g_plan.back();
  }
  return ATTN_OK;
}

// Grid of the forward when no balanced schedule is used (packed inputs, or a
// causal shape first seen while its stream is being captured). A persistent
// grid (one CTA per SM, static striding over the work list) overlaps
// consecutive tiles of a CTA, which saves the start-up and drain of a CTA per
// tile (taken as 2 us here; the gap between two CTAs on one SM measures about
// 4 us on GB300); one CTA per tile instead lets the
// hardware block scheduler balance unequal tiles greedily. Equal tiles (fixed
// length, no mask) always go persistent; otherwise persistence wins when the
// start-up it saves per SM outweighs the imbalance static striding can leave,
// at most about one longest tile (its key tiles times about 1.7 us at
// d_qk = d_v = 128, scaled by d_qk + d_v above that, and 0.9 us at 64, measured
// on GB300). Packed inputs use the mean length. `width` is d_qk + d_v.
bool fwd_persistent(long long tiles, int n_sm, bool causal, bool varlen, long long len, int width) {
  if (!causal && !varlen) return true;
  const double saved_us = 2.0 * static_cast<double>(tiles) / n_sm;
  const double per_key_tile_us = width <= 128 ? 0.9 : 1.7 * width / 256.0;
  const double longest_us = static_cast<double>((len + 127) / 128) * per_key_tile_us;
  return saved_us >= longest_us;
}

// Balanced persistent schedule of the forward for fixed-length inputs with
// unequal work tiles (causal masks): the work list, in its usual order, is
// dealt out greedily, each tile to the CTA with the least estimated work so
// far (longest-processing-time list scheduling; the order already runs the
// longest tiles of each L2 section first). A tile is estimated at the key tiles
// of its two query tiles plus a fixed cost of about six key tiles for its
// start and epilogue (measured on GB300). The lists depend only on the shape
// and the grid, are built on the host once per shape and kept on the device
// until the process exits, so a captured graph can keep using them.
int fwd_tile_units(long long v, int n_mblocks, int H_q, int sec_heads, int N_q, int N_k,
                   bool causal, int pair) {
  const int hu = H_q >> pair;  // heads in units of a work tile's heads
  const long long per_b = static_cast<long long>(n_mblocks) * hu;
  const int local = static_cast<int>(v % per_b);
  const int nm = n_mblocks;
  const int su = sec_heads >> pair;
  const int sec = local / (nm * su);
  const int r = local - sec * nm * su;
  const int u0 = sec * su;
  const int us = std::min(su, hu - u0);
  const int mi = r / us;
  const int m = causal ? (nm - 1 - mi) : mi;
  int units = 0;
  for (int i = 0; i < 2; ++i) {
    const int r0 = m * (256 >> pair) + (pair ? 0 : i * 128);
    if (r0 >= N_q) continue;
    int kv_end = N_k;
    if (causal) kv_end = std::min(kv_end, r0 + 128);
    units += (kv_end + 127) / 128;
  }
  return units;
}

constexpr long long kMaxListTiles = 1ll << 22;  // list of at most 16 MB

struct FwdSchedule {
  int dev, B, H_q, N_q, N_k, causal, sec_heads, grid, pair;
  int* ptr;  // cta_start [grid + 1] then tile_list [tiles]
};
std::mutex g_sched_mu;
std::vector<FwdSchedule> g_sched;

// Device copy of the balanced schedule; nullptr when it cannot be made now
// (while the stream is being captured, a new one is not built).
// The balanced lists on the host: cta_start [grid + 1] then tile_list [tiles].
std::vector<int> fwd_schedule_lists(int B, int H_q, int N_q, int N_k, bool causal, int sec_heads,
                                    int n_mblocks, int grid, int pair) {
  const long long tiles = static_cast<long long>(B) * n_mblocks * (H_q >> pair);
  constexpr long long kFixedUnits = 6;
  std::vector<int> owner(tiles), count(grid, 0);
  // min-heap of (estimated work, CTA)
  std::vector<std::pair<long long, int>> heap;
  heap.reserve(grid);
  for (int c = 0; c < grid; ++c) heap.emplace_back(0, c);
  auto later = [](const std::pair<long long, int>& a, const std::pair<long long, int>& b) {
    return a > b;
  };
  for (long long v = 0; v < tiles; ++v) {
    std::pop_heap(heap.begin(), heap.end(), later);
    auto& top = heap.back();
    owner[v] = top.second;
    ++count[top.second];
    top.first +=
        kFixedUnits + fwd_tile_units(v, n_mblocks, H_q, sec_heads, N_q, N_k, causal, pair);
    std::push_heap(heap.begin(), heap.end(), later);
  }
  std::vector<int> host(grid + 1 + tiles);
  host[0] = 0;
  for (int c = 0; c < grid; ++c) host[c + 1] = host[c] + count[c];
  std::vector<int> fill(host.begin(), host.begin() + grid);
  for (long long v = 0; v < tiles; ++v) host[grid + 1 + fill[owner[v]]++] = static_cast<int>(v);
  return host;
}

// Device copy of the balanced schedule; nullptr when it cannot be made now
// (while the stream is being captured, a new one is not built).
const int* fwd_schedule(int dev, cudaStream_t stream, int B, int H_q, int N_q, int N_k, bool causal,
                        int sec_heads, int n_mblocks, int grid, int pair) {
  std::lock_guard<std::mutex> lock(g_sched_mu);
  for (const FwdSchedule& f : g_sched)
    if (f.dev == dev && f.B == B && f.H_q == H_q && f.N_q == N_q && f.N_k == N_k &&
        f.causal == static_cast<int>(causal) && f.sec_heads == sec_heads && f.grid == grid &&
        f.pair == pair)
      return f.ptr;
  // at most kMaxSchedules shapes keep a list (they are never freed: a captured
  // graph may still use one); further shapes run one CTA per tile
  constexpr size_t kMaxSchedules = 256;
  if (g_sched.size() >= kMaxSchedules) return nullptr;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return nullptr;
  if (static_cast<long long>(B) * n_mblocks * (H_q >> pair) > kMaxListTiles) return nullptr;
  const std::vector<int> host =
      fwd_schedule_lists(B, H_q, N_q, N_k, causal, sec_heads, n_mblocks, grid, pair);
  // the copy completes before the schedule is shared: launches on other
  // streams may use it next
  void* ptr = nullptr;
  if (cudaMalloc(&ptr, host.size() * sizeof(int)) != cudaSuccess) return nullptr;
  if (cudaMemcpyAsync(ptr, host.data(), host.size() * sizeof(int), cudaMemcpyHostToDevice,
                      stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaFree(ptr);
    return nullptr;
  }
  g_sched.push_back(FwdSchedule{dev, B, H_q, N_q, N_k, causal ? 1 : 0, sec_heads, grid, pair,
                                static_cast<int*>(ptr)});
  return static_cast<int*>(ptr);
}

// Query heads per L2 section of the forward work list: as many whole KV-head
// groups as keep their K and V (rows x (d_qk + d_v) bf16 values) within a share
// of L2, cut evenly over the KV heads. `width` is d_qk + d_v.
int l2_section_heads(int H_q, int H_kv, long long rows, int width) {
  constexpr long long kBudget = 48ll << 20;
  const long long per_kv = rows * width * 2;
  long long fit = per_kv > 0 ? kBudget / per_kv : H_kv;
  if (fit < 1) fit = 1;
  if (fit > H_kv) fit = H_kv;
  const long long n_sec = (H_kv + fit - 1) / fit;
  const long long kv_per_sec = (H_kv + n_sec - 1) / n_sec;
  return static_cast<int>(kv_per_sec) * (H_q / H_kv);
}

// Launch plan of the forward: work tiles, L2 sections, and who takes which
// tile (kFwdOneCtaPerTile, kFwdStriding, kFwdBalancedList). The balanced list
// is the intent; a call falls back to one CTA per tile when the list cannot be
// made at that moment (stream capture of a new shape, or the shape cache full).
enum { kFwdOneCtaPerTile = 0, kFwdStriding = 1, kFwdBalancedList = 2, kFwdClaimed = 3 };
struct FwdPlan {
  long long tiles;  // exact for fixed length, an upper bound when packed
  int pair;         // work tiles of two query heads (causal, even GQA group)
  int n_mblocks;    // m-blocks (256 rows, 128 with pair) per batch entry (0 when packed)
  int sec_heads;
  int mode;
  long long grid;
};
FwdPlan fwd_plan(int B, int H_q, int H_kv, int N_q, int N_k, int d_qk, int d_v, bool causal,
                 bool varlen, int n_sm) {
  FwdPlan f;
  // work tiles: two 128-row query tiles, either 256 rows of one head or, under a
  // causal mask with an even GQA group, the same 128 rows of two heads of one KV
  // head. Exact for fixed length; for packed inputs an upper bound on the sum
  // over sequences of ceil(L / rows) times the head units.
  f.pair = (causal && (H_q / H_kv) % 2 == 0) ? 1 : 0;
  const long long mrows = 256 >> f.pair;
  const long long hu = H_q >> f.pair;
  f.tiles = varlen ? (static_cast<long long>(N_q) + (mrows - 1) * B) / mrows * hu
                   : static_cast<long long>(B) * ((N_q + mrows - 1) / mrows) * hu;
  f.n_mblocks = varlen ? 0 : static_cast<int>((N_q + mrows - 1) / mrows);
  // the mean sequence length sizes the L2 sections of packed inputs
  f.sec_heads = l2_section_heads(H_q, H_kv, varlen ? (N_k + B - 1) / B : N_k, d_qk + d_v);
  f.mode = kFwdOneCtaPerTile;
  f.grid = f.tiles;
  if (f.tiles > n_sm && varlen) {
    // packed: the tiles' sizes are known only on the device, so one CTA per SM
    // claims tiles from a counter as it finishes them (greedy list scheduling)
    f.mode = kFwdClaimed;
    f.grid = n_sm;
  } else if (f.tiles > n_sm) {
    if (fwd_persistent(f.tiles, n_sm, causal, varlen, varlen ? (N_k + B - 1) / B : N_k,
                       d_qk + d_v)) {
      f.mode = kFwdStriding;
      f.grid = n_sm;
    } else if (!varlen && f.tiles <= kMaxListTiles) {
      // long tiles of unequal, known size (causal masks)
      f.mode = kFwdBalancedList;
      f.grid = n_sm;
    }
  }
  return f;
}

// 4-D map over a [batch, rows, heads, d] bf16 tensor, one box = 128 (or
// box_rows) rows x 64 columns of one head, 128-byte swizzle (so the tile lands in shared memory in
// the layout the tcgen05 descriptors expect).
int encode_rows_map(CUtensorMap* m, const void* base, int d, int heads, long long rows,
                    long long batch, bool fp32 = false, unsigned box_rows = 128) {
  const cuuint64_t es_bytes = fp32 ? 4 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * es_bytes,
                           static_cast<cuuint64_t>(d) * es_bytes * heads,
                           static_cast<cuuint64_t>(d) * es_bytes * heads * rows};
  // 128 bytes of the innermost dimension per box row: 64 bf16 or 32 fp32
  cuuint32_t box[4] = {fp32 ? 32u : 64u, 1, box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        4, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

struct Shape {
  int B, H_q, H_kv, N_q, N_k, d;
  bool varlen;
  long long q_rows, k_rows;  // rows of the [rows, H, d] view (B*N fixed, T packed)
  long long q_batch;         // TMA batch extent (B fixed, 1 packed)
};

int check_shape(int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
                const int* seqlens, Shape* s) {
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  if (B < 0 || N_q < 0 || N_k < 0 || H_q <= 0 || H_kv <= 0) return ATTN_ERR_BAD_SHAPE;
  if (H_q % H_kv != 0) return ATTN_ERR_GQA_RATIO;
  if (H_q > 65535) return ATTN_ERR_BAD_SHAPE;
  s->B = B; s->H_q = H_q; s->H_kv = H_kv; s->N_q = N_q; s->N_k = N_k; s->d = d;
  s->varlen = seqlens != nullptr;
  if (s->varlen) {
    if (N_q != N_k) return ATTN_ERR_CAUSAL_SHAPE;  // one offset array for q and k/v
    if (B < 1) return ATTN_ERR_BAD_SHAPE;
    s->q_rows = N_q;
    s->k_rows = N_k;
    s->q_batch = 1;
  } else {
    if (causal && N_q != N_k) return ATTN_ERR_CAUSAL_SHAPE;
    if (B > 65535) return ATTN_ERR_BAD_SHAPE;
    s->q_rows = N_q;
    s->k_rows = N_k;
    s->q_batch = B;
  }
  // keep every element offset inside int64 and every TMA coordinate inside int32
  const long long elems = static_cast<long long>(B) * (N_q + N_k) * H_q * d;
  if (elems < 0 || elems > (1ll << 46)) return ATTN_ERR_BAD_SHAPE;
  return ATTN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// ---- kernel tracing: event pairs recorded around each launch
struct ProfSlot {
  int kernel;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfSlot> g_prof_open;   // recorded, not yet read
std::vector<cudaEvent_t> g_prof_free;

cudaEvent_t prof_event() {
  if (!g_prof_free.empty()) {
    cudaEvent_t e = g_prof_free.back();
    g_prof_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Workspace plan of the backward pass.
struct BwdPlan {
  long long rows_q;     // rows of the [rows, H_q, d] view of q
  long long slots;      // query-tile slots (deterministic semaphores), per head
  long long n_work;     // CTAs of the main kernel (upper bound for packed inputs)
  size_t acc_off, dvec_off, sem_off, order_off, total;
};

bool fwd_uses_pairs() {
  std::lock_guard<std::mutex> lock(g_mu);
  return g_fwd_variant == ATTN_FWD_CTA_PAIR;
}

// The d = 128 forward on CTA pairs: one cluster of two CTAs per 512 query rows
// of one (batch, query head); K is loaded in 64-row halves, one per CTA.
int fwd_pair(const CUtensorMap& tq, const void* k_base, int k_heads, long long k_rows,
             const CUtensorMap& tv, long long batch, void* o, float* lse, int B, int H_q,
             int H_kv, int N_q, int N_k, int causal, const int* seqlens, float scale, int* err,
             cudaStream_t cs) {
  CUtensorMap tk_half;
  if (encode_rows_map(&tk_half, k_base, 128, k_heads, k_rows, batch, false, 64u) != ATTN_OK)
    return ATTN_ERR_CUDA;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = seqlens;
  p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_k = N_k;
  p.group = H_q / H_kv;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * kLog2e;
  p.err = err;
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  constexpr long long kRows = 4 * kTileM;
  // packed: an upper bound on the sum over sequences of ceil(L / 512); the
  // pairs past the last block return at once
  const long long blocks = seqlens ? (static_cast<long long>(N_q) + (kRows - 1) * B) / kRows
                                   : (static_cast<long long>(N_q) + kRows - 1) / kRows;
  if (2 * blocks > 0x7fffffffll) return ATTN_ERR_BAD_SHAPE;
  const dim3 grid(static_cast<unsigned>(2 * blocks), static_cast<unsigned>(H_q),
                  seqlens ? 1u : static_cast<unsigned>(B));
  if (launch_attn_fwd_pair(tq, tk_half, tv, p, grid, cs) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

bool bwd_uses_pairs(int d) {
  std::lock_guard<std::mutex> lock(g_mu);
  return d == 128 && g_bwd_variant == ATTN_BWD_CTA_PAIR;
}

// The workspace size does not depend on `pairs` (only the work count does).
// `d` is the query/key head dimension (the width of the dQ accumulator); a
// query/key head dimension above 128 takes two passes of the main kernel, each
// with its own ordering semaphores in deterministic mode.
bool bwd_plan(int B, int H_q, int H_kv, int N_q, int N_k, int d, bool varlen, bool det,
              bool pairs, BwdPlan* pl) {
  const int passes = d > 128 ? 2 : 1;
  // work items: key tiles of 128 rows, or key pairs of 256 rows (one per CTA
  // pair)
  const long long kt = pairs ? 256 : 128;
  if (varlen) {
    pl->rows_q = N_q;
    pl->slots = (static_cast<long long>(N_q) + 127ll * B) / 128;
    pl->n_work = (static_cast<long long>(N_k) + (kt - 1) * B) / kt * H_kv;
  } else {
    pl->rows_q = static_cast<long long>(B) * N_q;
    pl->slots = static_cast<long long>(B) * ((N_q + 127) / 128);
    pl->n_work = static_cast<long long>(B) * H_kv * ((N_k + kt - 1) / kt);
  }
  if (pl->n_work > 0x7fffffffll || (pl->slots * H_q + 1) * passes > 0x7fffffffll) return false;
  pl->acc_off = 0;
  pl->dvec_off = align256(static_cast<size_t>(pl->rows_q) * H_q * d * 4);
  pl->sem_off = pl->dvec_off + align256(static_cast<size_t>(pl->rows_q) * H_q * 4);
  pl->order_off = pl->sem_off +
                  (det ? align256(static_cast<size_t>(pl->slots * H_q + 1) * passes * 4) : 0);
  // packed: the sequence order and the first work item of each sequence
  pl->total = pl->order_off + (varlen ? align256((2 * static_cast<size_t>(B) + 1) * 4) : 0);
  return true;
}

}  // namespace

namespace attn {
int prof_begin(int kernel, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof_on) return -1;
  ProfSlot s{kernel, prof_event(), prof_event()};
  if (!s.start || !s.stop) return -1;
  cudaEventRecord(s.start, stream);
  g_prof_open.push_back(s);
  return static_cast<int>(g_prof_open.size()) - 1;
}
void prof_end(int slot, cudaStream_t stream) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (slot < static_cast<int>(g_prof_open.size())) cudaEventRecord(g_prof_open[slot].stop, stream);
}
}  // namespace attn

extern "C" {

int attn_profile_enable(int enable) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = enable != 0;
  return ATTN_OK;
}

int attn_profile_read(attn_profile_record* out, int max_records) {
  if (max_records > 0 && out == nullptr) return -ATTN_ERR_NULL_PTR;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  int n = 0;
  for (const ProfSlot& s : g_prof_open) {
    if (cudaEventSynchronize(s.stop) != cudaSuccess) return -ATTN_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, s.start, s.stop) != cudaSuccess) return -ATTN_ERR_CUDA;
    if (n < max_records) out[n++] = attn_profile_record{s.kernel, ms};
    g_prof_free.push_back(s.start);
    g_prof_free.push_back(s.stop);
  }
  g_prof_open.clear();
  return n;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL_PTR: return "null pointer";
    case ATTN_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case ATTN_ERR_UNSUPPORTED_HEADDIM: return "unsupported head dimension (need 64 or 128)";
    case ATTN_ERR_BAD_SHAPE: return "invalid size or scalar argument";
    case ATTN_ERR_GQA_RATIO: return "H_q is not a multiple of H_kv";
    case ATTN_ERR_CAUSAL_SHAPE: return "N_q != N_k where they must match";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    case ATTN_ERR_NO_DEVICE: return "no usable CUDA device";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300 class)";
    case ATTN_ERR_SEQLENS: return "cu_seqlens is not 0, non-decreasing, ..., N_q";
    default: return "unknown status";
  }
}

int attn_set_bwd_variant(int variant) {
  if (variant != ATTN_BWD_ONE_CTA && variant != ATTN_BWD_CTA_PAIR) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  const int old = g_bwd_variant;
  g_bwd_variant = variant;
  return old;
}

int attn_set_fwd_variant(int variant) {
  if (variant != ATTN_FWD_ONE_CTA && variant != ATTN_FWD_CTA_PAIR) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  const int old = g_fwd_variant;
  g_fwd_variant = variant;
  return old;
}

long long attn_set_wait_limit(long long cycles) {
  std::lock_guard<std::mutex> lock(g_mu);
  const long long old = g_wait_limit.load();
  if (cycles > 0) g_wait_limit.store(cycles);
  return old;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
             int H_kv, int N_q, int N_k, int d, int causal, const int* seqlens, float scale,
             attn_stream_t stream) {
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  return attn_fwd_dims(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, d, causal, seqlens, scale,
                       stream);
}

int attn_fwd_dims(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int H_q, int H_kv, int N_q, int N_k, int d_qk, int d_v, int causal,
                  const int* seqlens, float scale, attn_stream_t stream) {
  if (!((d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128) || (d_qk == 192 && d_v == 128)))
    return ATTN_ERR_UNSUPPORTED_HEADDIM;
  Shape s;
  int st = check_shape(B, H_q, H_kv, N_q, N_k, d_v, causal, seqlens, &s);
  if (st != ATTN_OK) return st;
  // element-count bound of check_shape, with the wider head dimension
  if (static_cast<long long>(B) * (N_q + N_k) * H_q * d_qk > (1ll << 46)) return ATTN_ERR_BAD_SHAPE;
  // an empty tensor may come with a null pointer
  const bool has_q = B > 0 && N_q > 0, has_k = B > 0 && N_k > 0;
  if ((has_q && (!q || !o || !lse)) || (has_k && (!k || !v))) return ATTN_ERR_NULL_PTR;
  if (!std::isfinite(scale)) return ATTN_ERR_BAD_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (seqlens && (reinterpret_cast<uintptr_t>(seqlens) & 3u)))
    return ATTN_ERR_ALIGNMENT;
  if (B == 0 || N_q == 0) return ATTN_OK;
  int dev;
  if ((st = current_device(&dev)) != ATTN_OK) return st;
  int* err = nullptr;
  if ((st = device_setup(dev, &err)) != ATTN_OK) return st;

  CUtensorMap tq, tk, tv, to;
  // with no keys at all nothing is ever loaded from k/v; map q instead of an empty extent
  const bool no_keys = (N_k == 0);
  if (encode_rows_map(&tq, q, d_qk, H_q, s.q_rows, s.q_batch) != ATTN_OK ||
      encode_rows_map(&to, o, d_v, H_q, s.q_rows, s.q_batch) != ATTN_OK ||
      encode_rows_map(&tk, no_keys ? q : k, d_qk, no_keys ? H_q : H_kv,
                      no_keys ? s.q_rows : s.k_rows, s.q_batch) != ATTN_OK ||
      encode_rows_map(&tv, no_keys ? q : v, d_v, no_keys ? H_q : H_kv,
                      no_keys ? s.q_rows : s.k_rows, s.q_batch) != ATTN_OK)
    return ATTN_ERR_CUDA;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (d_qk == 128 && d_v == 128 && fwd_uses_pairs())
    return fwd_pair(tq, no_keys ? q : k, no_keys ? H_q : H_kv, no_keys ? s.q_rows : s.k_rows, tv,
                    s.q_batch, o, lse, B, H_q, H_kv, N_q, N_k, causal, seqlens, scale, err, cs);
  const int n_sm = sm_count(dev);
  if (n_sm <= 0) return ATTN_ERR_CUDA;
  const FwdPlan plan = fwd_plan(B, H_q, H_kv, N_q, N_k, d_qk, d_v, causal != 0,
                                seqlens != nullptr, n_sm);
  const long long tiles = plan.tiles;
  if (tiles > 0x7fffffffll) return ATTN_ERR_BAD_SHAPE;

  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = seqlens;
  p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_k = N_k;
  p.group = H_q / H_kv;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * kLog2e;
  p.err = err;
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  p.seq_order = nullptr;
  p.tile_start = nullptr;
  p.tile_list = nullptr;
  p.cta_start = nullptr;
  p.tile_ctr = nullptr;
  p.total_tiles = static_cast<int>(tiles);
  p.n_mblocks = plan.n_mblocks;
  p.pair_heads = plan.pair;
  p.sec_heads = plan.sec_heads;
  if (seqlens) {
    PlanBuf pb;
    if ((st = plan_buffer(dev, cs, B, &pb)) != ATTN_OK) return st;
    int* order = pb.ptr;
    int* start = order + pb.cap;
    int* ctr = start + pb.cap + 1;
    if (launch_fwd_plan(seqlens, B, N_q, H_q, p.pair_heads, order, start, ctr, err, cs) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    p.seq_order = order;
    p.tile_start = start;
    p.n_mblocks = 0;  // per sequence
    if (plan.mode == kFwdClaimed) p.tile_ctr = ctr;
  }
  long long grid_x = tiles;
  if (plan.mode == kFwdStriding || plan.mode == kFwdClaimed) {
    grid_x = plan.grid;
  } else if (plan.mode == kFwdBalancedList) {
    const int* sch = fwd_schedule(dev, cs, B, H_q, N_q, N_k, causal != 0, p.sec_heads,
                                  p.n_mblocks, n_sm, plan.pair);
    if (sch) {
      p.cta_start = sch;
      p.tile_list = sch + n_sm + 1;
      grid_x = plan.grid;
    }
  }
  if (launch_attn_fwd(d_qk, d_v, tq, tk, tv, to, p, dim3(static_cast<unsigned>(grid_x)), cs) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

size_t attn_bwd_workspace_bytes(int B, int H_q, int H_kv, int N_q, int N_k, int d, int varlen,
                                int deterministic) {
  if (d != 64 && d != 128) return 0;
  return attn_bwd_dims_workspace_bytes(B, H_q, H_kv, N_q, N_k, d, d, varlen, deterministic);
}

namespace {
bool bwd_dims_supported(int d_qk, int d_v) {
  return (d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128) || (d_qk == 192 && d_v == 128);
}
}  // namespace

size_t attn_bwd_dims_workspace_bytes(int B, int H_q, int H_kv, int N_q, int N_k, int d_qk, int d_v,
                                     int varlen, int deterministic) {
  if (!bwd_dims_supported(d_qk, d_v)) return 0;
  Shape s;
  if (check_shape(B, H_q, H_kv, N_q, N_k, d_v, 0, varlen ? reinterpret_cast<const int*>(16) : nullptr,
                  &s) != ATTN_OK)
    return 0;
  if (static_cast<long long>(B) * (N_q + N_k) * H_q * d_qk > (1ll << 46)) return 0;
  BwdPlan pl;
  if (!bwd_plan(B, H_q, H_kv, N_q, N_k, d_qk, varlen != 0, deterministic != 0, false, &pl)) return 0;
  return pl.total;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int N_q,
             int N_k, int d, int causal, const int* seqlens, float scale, int deterministic,
             void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  return attn_bwd_dims(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d, d, causal,
                       seqlens, scale, deterministic, workspace, workspace_bytes, stream);
}

int attn_bwd_dims(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, int B, int H_q, int H_kv,
                  int N_q, int N_k, int d_qk, int d_v, int causal, const int* seqlens, float scale,
                  int deterministic, void* workspace, size_t workspace_bytes,
                  attn_stream_t stream) {
  if (!bwd_dims_supported(d_qk, d_v)) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  Shape s;
  int st = check_shape(B, H_q, H_kv, N_q, N_k, d_v, causal, seqlens, &s);
  if (st != ATTN_OK) return st;
  // element-count bound of check_shape, with the wider head dimension
  if (static_cast<long long>(B) * (N_q + N_k) * H_q * d_qk > (1ll << 46)) return ATTN_ERR_BAD_SHAPE;
  const bool has_q = B > 0 && N_q > 0, has_k = B > 0 && N_k > 0;
  if ((has_q && (!q || !o || !lse || !dout || !dq)) || (has_k && (!k || !v || !dk || !dv)))
    return ATTN_ERR_NULL_PTR;
  if (!std::isfinite(scale)) return ATTN_ERR_BAD_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (seqlens && (reinterpret_cast<uintptr_t>(seqlens) & 3u)))
    return ATTN_ERR_ALIGNMENT;
  BwdPlan pl;
  const bool pairs = d_qk == d_v && bwd_uses_pairs(d_qk);
  if (!bwd_plan(B, H_q, H_kv, N_q, N_k, d_qk, seqlens != nullptr, deterministic != 0, pairs, &pl))
    return ATTN_ERR_BAD_SHAPE;
  if (B == 0) return ATTN_OK;
  const bool empty = (N_q == 0 || N_k == 0);
  if (!empty && (workspace == nullptr || workspace_bytes < pl.total)) return ATTN_ERR_WORKSPACE;
  if (!empty && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_ALIGNMENT;
  int dev;
  if ((st = current_device(&dev)) != ATTN_OK) return st;
  int* err = nullptr;
  if ((st = device_setup(dev, &err)) != ATTN_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t k_rows = static_cast<size_t>(s.varlen ? N_k : static_cast<long long>(B) * N_k);
  const size_t q_bytes = static_cast<size_t>(pl.rows_q) * H_q * d_qk * 2;
  const size_t k_bytes = k_rows * H_kv * d_qk * 2;
  const size_t v_bytes = k_rows * H_kv * d_v * 2;
  if (empty) {
    // no query rows: no key gradient; no keys: every row sees nothing
    if ((q_bytes && cudaMemsetAsync(dq, 0, q_bytes, cs) != cudaSuccess) ||
        (k_bytes && cudaMemsetAsync(dk, 0, k_bytes, cs) != cudaSuccess) ||
        (v_bytes && cudaMemsetAsync(dv, 0, v_bytes, cs) != cudaSuccess))
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // q, k (d_qk), v, dO (d_v) with 128-row boxes, the fp32 dQ accumulator
  // (d_qk; 128-row boxes, 64 on CTA pairs), and on CTA pairs q and dO with
  // 64-row boxes
  CUtensorMap maps[9];
  if (encode_rows_map(&maps[0], q, d_qk, H_q, s.q_rows, s.q_batch) != ATTN_OK ||
      encode_rows_map(&maps[1], k, d_qk, H_kv, s.k_rows, s.q_batch) != ATTN_OK ||
      encode_rows_map(&maps[2], v, d_v, H_kv, s.k_rows, s.q_batch) != ATTN_OK ||
      encode_rows_map(&maps[3], dout, d_v, H_q, s.q_rows, s.q_batch) != ATTN_OK ||
      encode_rows_map(&maps[4], ws + pl.acc_off, d_qk, H_q, s.q_rows, s.q_batch, true,
                      pairs ? 64u : 128u) != ATTN_OK)
    return ATTN_ERR_CUDA;
  if (pairs && (encode_rows_map(&maps[5], q, d_qk, H_q, s.q_rows, s.q_batch, false, 64u) != ATTN_OK ||
                encode_rows_map(&maps[6], dout, d_v, H_q, s.q_rows, s.q_batch, false, 64u) != ATTN_OK))
    return ATTN_ERR_CUDA;
  // dK and dV, written by TMA stores from the one-CTA kernel's epilogue
  if (encode_rows_map(&maps[7], dk, d_qk, H_kv, s.k_rows, s.q_batch) != ATTN_OK ||
      encode_rows_map(&maps[8], dv, d_v, H_kv, s.k_rows, s.q_batch) != ATTN_OK)
    return ATTN_ERR_CUDA;

  BwdParams p;
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.dout = dout;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.dq_acc = reinterpret_cast<float*>(ws + pl.acc_off);
  p.dvec = reinterpret_cast<float*>(ws + pl.dvec_off);
  p.sem = deterministic ? reinterpret_cast<int*>(ws + pl.sem_off) : nullptr;
  p.cu_seqlens = seqlens;
  p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_k = N_k; p.group = H_q / H_kv;
  p.d = d_qk;
  p.d_v = d_v;
  p.causal = causal ? 1 : 0;
  p.deterministic = deterministic ? 1 : 0;
  p.n_nblocks = 0;
  p.n_mtiles = 0;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.err = err;
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  p.fault = g_fault.load(std::memory_order_relaxed);
  p.pairs = pairs ? 1 : 0;
  p.sem_slots = static_cast<int>(pl.slots);
  p.seq_order = nullptr;
  p.item_start = nullptr;
  p.sec_heads = 0;
  // only for long items (at least 32 key tiles a pair): the longest item is
  // then a sizeable share of an SM's work, while with short items the pairs'
  // shared Q, dO and dQ rows in L2 are worth more than the balance
  if (causal && !seqlens && !pairs && (N_k + kTileN - 1) / kTileN >= 32) {
    // (batch, KV head) pairs per section: as many as keep what their items
    // stream within 48 MiB of L2: the GQA group's Q and dO (bf16, d_qk + d_v
    // values a row) and its fp32 dQ accumulator (d_qk values a row)
    constexpr long long kBudget = 48ll << 20;
    const long long per_pair =
        static_cast<long long>(N_q) * (H_q / H_kv) * (2ll * (d_qk + d_v) + 4ll * d_qk);
    long long fit = per_pair > 0 ? kBudget / per_pair : 1;
    if (fit < 1) fit = 1;
    if (fit > static_cast<long long>(B) * H_kv) fit = static_cast<long long>(B) * H_kv;
    p.sec_heads = static_cast<int>(fit);
  }
  if (seqlens && !pairs) {
    // packed: the work items walk the sequences longest first (greedy dispatch
    // of unequal items then ends with the short ones)
    int* order = reinterpret_cast<int*>(ws + pl.order_off);
    int* start = order + B;
    if (launch_seq_plan(seqlens, B, N_q, kTileN, H_kv, order, start, nullptr, err, kKBwdPlan, cs) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    p.seq_order = order;
    p.item_start = start;
  }
  // Deterministic order of the dQ additions: under a causal mask, and without
  // one when queries and keys have equal lengths and the key tiles of a (batch,
  // KV head) are few (non-causal key tiles wait on one another in a cycle, so
  // they must be resident together: at most 32, and at most one per SM), the
  // step order that keeps key tiles from stalling; otherwise ascending key
  // tiles. Packed sequences share q and k lengths; their key tiles per sequence
  // are at most those of all rows together.
  p.spt = 0;
  if (deterministic && !pairs) {
    const int n_sm = sm_count(dev);
    if (n_sm <= 0) return ATTN_ERR_CUDA;
    const long long nk = (static_cast<long long>(N_k) + kTileN - 1) / kTileN;
    p.spt = (causal || ((seqlens || N_q == N_k) && nk <= n_sm && nk <= 32)) ? 1 : 0;
  }
  const int n_sem = static_cast<int>(pl.slots * H_q);
  if (launch_attn_bwd(p, maps, cs, pl.rows_q, n_sem, static_cast<int>(pl.n_work)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

int attn_check(attn_stream_t stream) {
  int dev;
  int st = current_device(&dev);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  int* err = nullptr;
  if ((st = device_setup(dev, &err)) != ATTN_OK) return st;
  int h = 0;
  if (cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return h == kErrSeqlens ? ATTN_ERR_SEQLENS : ATTN_ERR_TIMEOUT;
  }
  return ATTN_OK;
}

int attn_debug_fwd_plan(int B, int H_q, int H_kv, int N_q, int N_k, int d_qk, int d_v,
                        int causal, int varlen, int n_sm, long long* info, int* lists,
                        long long lists_cap) {
  if (info == nullptr || n_sm <= 0) return ATTN_ERR_NULL_PTR;
  if (!((d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128) || (d_qk == 192 && d_v == 128)))
    return ATTN_ERR_UNSUPPORTED_HEADDIM;
  Shape s;
  const int st = check_shape(B, H_q, H_kv, N_q, N_k, d_v, causal,
                             varlen ? reinterpret_cast<const int*>(16) : nullptr, &s);
  if (st != ATTN_OK) return st;
  if (static_cast<long long>(B) * (N_q + N_k) * H_q * d_qk > (1ll << 46)) return ATTN_ERR_BAD_SHAPE;
  const FwdPlan f = fwd_plan(B, H_q, H_kv, N_q, N_k, d_qk, d_v, causal != 0, varlen != 0, n_sm);
  info[0] = f.mode;
  info[1] = f.grid;
  info[2] = f.tiles;
  info[3] = f.sec_heads;
  info[4] = f.n_mblocks;
  info[5] = f.pair;
  if (f.mode == kFwdBalancedList && lists != nullptr && lists_cap >= f.grid + 1 + f.tiles) {
    const std::vector<int> h = fwd_schedule_lists(B, H_q, N_q, N_k, causal != 0, f.sec_heads,
                                                  f.n_mblocks, static_cast<int>(f.grid), f.pair);
    std::memcpy(lists, h.data(), h.size() * sizeof(int));
  }
  return ATTN_OK;
}

int attn_debug_inject(int fault) {
  if (fault != ATTN_FAULT_NONE && fault != ATTN_FAULT_SKIP_DQ_RELEASE) return ATTN_ERR_BAD_SHAPE;
  std::lock_guard<std::mutex> lock(g_mu);
  g_fault.store(fault);
  return ATTN_OK;
}

int attn_debug_stall(attn_stream_t stream) {
  int dev;
  int st = current_device(&dev);
  if (st != ATTN_OK) return st;
  int* err;
  if ((st = device_setup(dev, &err)) != ATTN_OK) return st;
  return launch_stall_probe(err, g_wait_limit.load(std::memory_order_relaxed),
                            reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

int attn_debug_rescale_stats(unsigned long long* out, int reset) {
  if (out == nullptr) return -ATTN_ERR_NULL_PTR;
  int dev;
  const int st = current_device(&dev);
  if (st != ATTN_OK) return -st;
  const int n = read_rescale_stats(out, reset);
  return n < 0 ? -ATTN_ERR_CUDA : n;
}

int attn_debug_exp2(const float* x, float* y, int n, int mode, attn_stream_t stream) {
  if (n < 0) return ATTN_ERR_BAD_SHAPE;
  if (n > 0 && (!x || !y)) return ATTN_ERR_NULL_PTR;
  int dev;
  int st = current_device(&dev);
  if (st != ATTN_OK) return st;
  int* err;
  if ((st = device_setup(dev, &err)) != ATTN_OK) return st;
  return launch_exp2_probe(x, y, n, mode ? 1 : 0, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

}  // extern "C"

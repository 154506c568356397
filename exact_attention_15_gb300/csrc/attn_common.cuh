// Shared definitions of the attention kernels: launch parameters, tile sizes,
// the FMA-pipe exp2 and the device error word.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace attn {

constexpr int kTileM = 128;   // query rows per tile (tcgen05 M)
constexpr int kTileN = 128;   // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Conditional rescaling threshold, in powers of two: the running max used for
// the exponentials is only moved when the true max has grown by more than
// 2^8 = 256 (FlashAttention-4 summary, section 3.1.4). A measurement build may
// set ATTN_TAU (0 rescales whenever the max grows, the baseline the pages
// compare against); results differ only by rounding.
#ifndef ATTN_TAU
#define ATTN_TAU 8.0f
#endif
constexpr float kTau = ATTN_TAU;
// ATTN_COUNT_RESCALE = 1 builds counters of the forward's rescale events
// (attn_debug_rescale_stats); the shipped build has none.
#ifndef ATTN_COUNT_RESCALE
#define ATTN_COUNT_RESCALE 0
#endif

// Device error word values (the first failure is kept): a bounded wait ran
// out; a packed-sequence offset array is not 0, non-decreasing, ..., T.
enum DevErr : int { kErrNone = 0, kErrTimeout = 1, kErrSeqlens = 2 };
// Host-injected faults (attn_debug_inject); none of them can fault or hang the GPU.
enum Fault : int { kFaultNone = 0, kFaultSkipDqRelease = 1 };

struct FwdParams {
  void* o;              // bf16
  float* lse;
  const int* cu_seqlens;  // nullptr for fixed length
  int B, H_q, H_kv, N_q, N_k, group;
  int causal;
  int n_mblocks;        // m-blocks per batch entry (fixed length only): 256 query rows, or
                        // 128 with pair_heads
  int pair_heads;       // 1: a work tile is the same 128 query rows of two adjacent query
                        // heads of one KV head (causal, even GQA group); 0: 256 rows of one head
  float scale_log2;     // scale * log2(e)
  int* err;             // device error word
  long long wait_limit; // cycles
  // Work list of the forward (longest-processing-time-first order).
  const int* tile_list;   // balanced schedule: work tiles of CTA c are
  const int* cta_start;   //   tile_list[cta_start[c] .. cta_start[c + 1]) (nullptr: striding)
  int* tile_ctr;          // claimed schedule: claim counter, zero at launch (nullptr: static)
  const int* seq_order;   // packed: virtual -> actual sequence, longest first
  const int* tile_start;  // packed: first work tile of each virtual sequence, [B + 1]
  int total_tiles;        // fixed length: B * n_mblocks * (H_q >> pair_heads)
  int sec_heads;          // query heads per L2 section (a multiple of H_q / H_kv)
};

struct BwdParams {
  const void* q; const void* k; const void* v; const void* o; const float* lse;
  const void* dout;
  void* dq; void* dk; void* dv;
  float* dq_acc;        // fp32 [rows, H_q, d]
  float* dvec;          // fp32 D, laid out like lse
  int* sem;             // deterministic mode: one counter per (b, h_q, query tile)
  const int* cu_seqlens;
  int B, H_q, H_kv, N_q, N_k, group, d;  // d: query/key head dimension
  int d_v;                               // value head dimension
  int causal, deterministic;
  int n_nblocks;        // key tiles per (batch, kv head) or upper bound (packed)
  int n_mtiles;         // query tiles per (batch, head) (fixed length) or upper bound
  float scale, scale_log2;
  int* err;
  long long wait_limit;
  int fault;            // host-injected fault for failure tests (0 = none)
  int pairs;            // d = 128: run the CTA-pair main kernel
  int spt;              // deterministic one-CTA kernel: key tiles in descending order,
                        // query tiles walked from the key tile's own, dQ added in step order
  // packed inputs, one-CTA kernels: the work items walk the sequences longest
  // first (seq_order: virtual -> actual sequence; item_start[v]: first item of
  // virtual sequence v, B + 1 entries); nullptr: input order
  const int* seq_order;
  const int* item_start;
  int sem_slots;        // query-tile slots per head the semaphore array holds
  int sec_heads;        // fixed length, causal: (batch, KV head) pairs per L2 section whose
                        // items run key tile major; 0: each pair's key tiles in a row
};

// Kernel tracing (host side, implemented next to the C ABI). prof_begin
// returns a slot (or -1 when tracing is off); prof_end closes it.
enum KernelId : int { kKFwd = 1, kKBwdPre = 2, kKBwdMain = 3, kKBwdPost = 4, kKExp2 = 5,
                      kKStall = 6, kKFwdPlan = 7, kKFwdPair = 8, kKBwdMain2 = 9,
                      kKBwdPlan = 10 };
int prof_begin(int kernel, cudaStream_t stream);
void prof_end(int slot, cudaStream_t stream);

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Byte offset inside a 128-byte-swizzled [rows x 64 bf16] block of element
// (row, col): the 16-byte chunk index is XORed with row % 8.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk16) {
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk16 ^ (row & 7)) << 4));
}

// Records the first device-side failure; never traps.
__device__ __forceinline__ void record_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// Rows [start, start + len) of packed sequence s, read from cu_seqlens and
// clamped so that they always lie inside the T packed rows the tensors hold,
// whatever the array contains: start = clamp(cu[s], lo, T), end =
// clamp(cu[s + 1], start, T). With lo = 0 each sequence is clamped on its own;
// a caller that walks the sequences in order passes the previous sequence's
// end as lo, which also keeps the spans disjoint and their total within T. A
// valid array (cu[0] = 0, non-decreasing, cu[B] = T) is returned unchanged;
// check_cu_seqlens reports an invalid one.
struct SeqSpan {
  int start, len;
};
__device__ __forceinline__ SeqSpan seq_span(const int* cu, int s, int T, int lo) {
  const int a = min(max(__ldg(cu + s), lo), T);
  const int e = min(max(__ldg(cu + s + 1), a), T);
  return SeqSpan{a, e - a};
}

// Records kErrSeqlens unless cu[0] = 0, cu[s] <= cu[s + 1] and cu[B] = T;
// thread `tid` of `nthreads` checks its share of the B + 1 entries.
__device__ __forceinline__ void check_cu_seqlens(const int* cu, int B, int T, int* err,
                                                 long long tid, long long nthreads) {
  for (long long s = tid; s <= B; s += nthreads) {
    const int c = __ldg(cu + s);
    const bool bad = (s == 0 && c != 0) || (s == B && c != T) || (s < B && c > __ldg(cu + s + 1));
    if (bad) record_error(err, kErrSeqlens);
  }
}

// 2^x on the FMA pipe for a pair of values, with packed fp32 instructions
// (about five instructions per value): Cody-Waite split x = floor(x) + f, f in
// [0, 1), by a round-down add of 2^23 + 2^22; a degree-3 minimax polynomial for
// 2^f (coefficients fitted by fit_exp2_poly.py, max relative error 8.6e-5 on
// [0, 1)); and the integer part added straight into the exponent field
// (FlashAttention-4 summary, 3.1.3) as t_bits << 23, which equals floor(x) << 23
// modulo 2^32 because the low 22 bits of the shift constant's encoding are 0.
// x is clamped at -127 so the exponent arithmetic cannot underflow; callers
// must not pass -inf for an element that has to come out as exactly 0.
__device__ __forceinline__ void exp2_poly3_x2(float x0, float x1, float& y0, float& y1) {
  constexpr float kC1 = 0.6951167583465576f;
  constexpr float kC2 = 0.22764499485492706f;
  constexpr float kC3 = 0.07706703990697861f;
  constexpr float kShift = 12582912.0f;  // 2^23 + 2^22
  const uint64_t sh = f32x2(kShift, kShift);
  const uint64_t x = f32x2(fmaxf(x0, -127.0f), fmaxf(x1, -127.0f));
  const uint64_t t = add_rm_f32x2(x, sh);          // kShift + floor(x), exactly
  const uint64_t f = sub_f32x2(x, sub_f32x2(t, sh));  // fraction in [0, 1)
  uint64_t p = fma_f32x2(f32x2(kC3, kC3), f, f32x2(kC2, kC2));
  p = fma_f32x2(p, f, f32x2(kC1, kC1));
  p = fma_f32x2(p, f, f32x2(1.0f, 1.0f));
  float p0, p1, t0, t1;
  f32x2_split(p, p0, p1);
  f32x2_split(t, t0, t1);
  y0 = __int_as_float(__float_as_int(p0) + (__float_as_int(t0) << 23));
  y1 = __int_as_float(__float_as_int(p1) + (__float_as_int(t1) << 23));
}

}  // namespace attn

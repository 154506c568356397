// Forward pass of exact softmax attention for sm_103a.
//
// A work tile is two 128-row query tiles of one (batch, query head); the CTA
// that owns it streams every key/value tile they see through shared memory
// (FlashAttention-4 summary, section 3.1.2: two output tiles per CTA, one
// softmax warpgroup per tile, one thread per row; the FlashAttention-2 loop order
// with the query tile outside and keys/values inside). Work tiles are numbered
// in longest-processing-time-first order (section 3.3) and CTA c takes tiles
// c, c + gridDim.x, c + 2 gridDim.x, ... The host picks the grid: one CTA per
// work tile when tile lengths differ (causal masks, packed sequences), so the
// hardware block scheduler hands the tiles out greedily in LPT order; one CTA
// per SM when they are all equal, so consecutive tiles of a CTA overlap (the
// next tile's Q and K/V loads and first S MMAs run under the current tile's
// last P V MMAs and epilogue).
//
// Warp roles (384 threads):
//   warp 0      TMA producer: both Q tiles of a work tile, then K_j / V_j into a
//               ring of single-tile stages (order K0 V0 K1 V1 ...).
//   warp 1      TMEM owner and MMA issuer (one thread): S_t = Q_t K_j^T (SS) and
//               O_t += P_t V_j (TS, P read from TMEM), ping-ponging the tiles so
//               the tensor core works on one tile while the other is in softmax.
//   warps 4-7   softmax for tile 0, warps 8-11 softmax for tile 1: load the S row
//               from TMEM, mask, row max, conditional rescale (tau = 8 in powers
//               of two, decided per warp), exp2, row sum, P (bf16) back into the S
//               columns of TMEM, and finally the epilogue O / l and LSE.
// Every role derives the work tile from (blockIdx.x, k) itself; nothing about
// the work list passes between roles.
//
// TMEM (512 columns): O_0 [0, d), O_1 [d, 2d), S_0/P_0 [2d, 2d+128),
// S_1/P_1 [2d+128, 2d+256).
#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "fwd_softmax.cuh"

namespace attn {

// P can go to the tensor core in two stages (FlashAttention-4 summary, section
// 3.1.2): the softmax warpgroup stores the first kPWords0 packed words of each
// row (keys [0, 2 kPWords0)), signals p_part, and the MMA warp starts O += P V
// on those keys while the rest of the row is exponentiated; p_full covers the
// remaining words. 48 words = three quarters of the 128 keys = 6 of the 8
// K-steps of the PV MMA; 64 stores P in one piece. Measured on GB300 the staged
// store is 2-3% slower on every workload (the extra barrier costs the issuing
// thread more than an earlier start of PV gains while the other query tile's
// MMAs keep the tensor core busy), so one piece is the default.
#ifndef ATTN_FWD_P_WORDS0
#define ATTN_FWD_P_WORDS0 64
#endif
constexpr int kPWords0 = ATTN_FWD_P_WORDS0;
static_assert(kPWords0 == 48 || kPWords0 == 64, "P split: three quarters or none");
constexpr int kPvSteps0 = kPWords0 / 8;  // PV K-steps (16 keys each) on the first part

#if ATTN_COUNT_RESCALE
// [0] (warp, key tile) softmax steps after a row's first key tile, [1] those
// steps in which the warp rescaled (some row's bias moved), [2] rows whose
// bias moved, [3] row steps counted
__device__ unsigned long long g_rescale_stats[4];
#endif

// Shared-memory plan. Q/K rows have DQK columns, V/O rows DV columns; every
// tile is stored as 128-row x 64-column (16 KB) 128-byte-swizzled blocks.
// Equal head dimensions: K and V share a ring of single-tile stages (load order
// K0 V0 K1 V1 ...). DQK != DV (192 / 128): K and V tiles differ in size, and
// two Q tiles plus stages of the larger tile do not fit, so the ring is made of
// 16 KB block slots instead: K_j takes DQK / 64 consecutive slots, V_j DV / 64.
template <int DQK, int DV>
struct FwdCfg {
  static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= 128, "head dimensions");
  static constexpr int kQBlocks = DQK / 64;              // column blocks of a Q or K tile
  static constexpr int kVBlocks = DV / 64;               // column blocks of a V tile
  static constexpr int kBlockBytes = kTileM * 64 * 2;    // 16 KB
  static constexpr int kQTileBytes = kQBlocks * kBlockBytes;
  static constexpr bool kBlockRing = DQK != DV;
  static constexpr int kTileBytes = kQTileBytes;         // one K or V stage (equal dims)
  static constexpr int kStages = kBlockRing ? 1 : (DQK == 128 ? 4 : 8);
  static constexpr int kSlots = 8;                       // block ring
  static constexpr int kFullBars = 4;                    // block ring: loads in flight <= 8 / 2
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kQTileBytes;
  static constexpr int kRingBytes = kBlockRing ? kSlots * kBlockBytes : kStages * kTileBytes;
  static constexpr int kBarOff = kKVOff + kRingBytes;
  // Equal head dimensions leave room for one 16 KB staging buffer per softmax
  // warpgroup: O can leave through shared memory and TMA stores (whole 128-byte
  // rows) instead of each thread storing its own row (kernels that use it ask
  // for kSmemBytesEpi).
  static constexpr bool kTmaEpi = DQK == DV;
  static constexpr int kOEpiOff = kBarOff + 1024;  // 1024-aligned for the 128-byte swizzle
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // barriers + alignment slack
  static constexpr int kSmemBytesEpi = kTmaEpi ? kOEpiOff + 2 * kBlockBytes + 1024 : kSmemBytes;
  static constexpr uint32_t kColO0 = 0, kColO1 = DV;
  static constexpr uint32_t kColS0 = 2 * DV, kColS1 = 2 * DV + 128;
  // d = 64: O (64 columns each) leaves room for P in its own columns (bf16
  // pairs, 64 each) beside S, so S of the next key tile can be computed while
  // the softmax still turns the current one into P; otherwise P overwrites S.
  static constexpr bool kSepP = DQK == 64 && DV == 64;
  static constexpr uint32_t kColP0 = kSepP ? 2 * DV + 256 : kColS0;
  static constexpr uint32_t kColPStep = kSepP ? 64 : 128;  // P_1 = P_0 + kColPStep
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 232448 && kSmemBytesEpi <= 232448, "shared memory");
  static_assert(kOEpiOff % 1024 == 0, "staging buffer alignment");
};

// Work decode: one work tile = two 128-row query tiles of one (batch, query head).
struct __align__(16) FwdTile {
  int b, h, h_kv;  // b < 0 marks the end of the work list
  int q0;          // first query row of tile 0, relative to the sequence
  int row_base;    // global packed-row offset of the sequence (0 for fixed length)
  int batch_coord; // TMA batch coordinate (b for fixed length, 0 for packed)
  int Lq, Lk;
  int n[2];        // key tiles each query tile visits
  int valid[2];
};

// Where a work tile lies: its sequence (batch entry) and its index within that
// sequence's tiles.
struct FwdWork {
  int local;     // tile index within the sequence; < 0 marks the end of the list
  int b;         // batch entry or packed sequence
  int row_base;  // first packed row of the sequence (0 for fixed length)
  int L;         // sequence length (fixed length: N_q)
};

// Slots of the ring through which the scheduler warp hands the decoded work
// tiles to the other roles, and the readers of each slot (the producer
// thread, the MMA warp and the eight softmax warps).
constexpr int kSchedSlots = 2;
constexpr int kSchedReaders = 10;
struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t s_full[2];
  uint64_t p_part[2];   // the first kPWords0 packed P words of the row are in TMEM
  uint64_t p_full[2];   // all of P is in TMEM
  uint64_t pv_done[2];   // O_t complete (last PV of a tile; every PV with a separate P)
  uint64_t s_free[2];    // separate P: the softmax has S_t in registers
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  // work tiles handed out by the scheduler warp
  uint64_t sched_full[kSchedSlots];
  uint64_t sched_empty[kSchedSlots];
  int sched_taken;     // work tiles the producer has taken so far
  FwdTile sched_t[kSchedSlots];
  uint32_t tmem_base;
};
// Longest-processing-time-first order of the work list (FlashAttention-4
// summary, section 3.3). The batch (for packed inputs: the sequence, taken
// longest first through seq_order) is outermost; inside it the query heads are
// cut into sections whose K/V fit in L2; inside a section the m-blocks run
// longest first (reversed for causal masks) and the heads of the section are
// innermost, so all query heads of a KV head are visited before the next
// m-block. locate_fwd_work finds the sequence of work tile v; expand_fwd_work
// finds the head and m-block inside it.
__device__ __forceinline__ FwdWork locate_fwd_work(const FwdParams& p, int v) {
  FwdWork w;
  if (p.cu_seqlens == nullptr) {
    const int per_b = p.n_mblocks * (p.H_q >> p.pair_heads);
    w.b = v / per_b;
    w.local = v - w.b * per_b;
    w.row_base = 0;
    w.L = p.N_q;
  } else {
    // largest virtual sequence whose first tile is <= v (sequences without
    // tiles share their start with the next one and are never selected)
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.tile_start[mid] <= v) lo = mid; else hi = mid;
    }
    w.b = p.seq_order[lo];
    w.local = v - p.tile_start[lo];
    const SeqSpan sp = seq_span(p.cu_seqlens, w.b, p.N_q, 0);
    w.row_base = sp.start;
    w.L = sp.len;
  }
  return w;
}

// Query tile i of a work tile: rows q0 + 128 i of head h, or, with pair_heads,
// rows q0 of head h + i. Under a causal mask the head pairs give both query
// tiles the same key tiles, so neither softmax warpgroup waits out the other's
// extra diagonal tile at the end of a work tile.
__device__ __forceinline__ int qtile_row(const FwdParams& p, const FwdTile& t, int i) {
  return t.q0 + (p.pair_heads ? 0 : i * kTileM);
}
__device__ __forceinline__ int qtile_head(const FwdParams& p, const FwdTile& t, int i) {
  return t.h + (p.pair_heads ? i : 0);
}

__device__ __forceinline__ void expand_fwd_work(const FwdParams& p, const FwdWork& w, FwdTile& t) {
  t.b = w.b;
  t.row_base = w.row_base;
  t.batch_coord = p.cu_seqlens ? 0 : w.b;
  t.Lq = w.L;
  t.Lk = p.cu_seqlens ? w.L : p.N_k;
  // heads in units of the heads of one work tile (1, or 2 with pair_heads)
  const int pr = p.pair_heads;
  const int mrows = (2 * kTileM) >> pr;
  const int nm = (w.L + mrows - 1) / mrows;
  const int su = p.sec_heads >> pr;
  const int sec = w.local / (nm * su);
  const int r = w.local - sec * nm * su;
  const int u0 = sec * su;
  const int us = min(su, (p.H_q >> pr) - u0);
  const int mi = r / us;
  t.h = (u0 + (r - mi * us)) << pr;
  t.h_kv = t.h / p.group;
  const int m = p.causal ? (nm - 1 - mi) : mi;
  t.q0 = m * mrows;
  for (int i = 0; i < 2; ++i) {
    const int r0 = qtile_row(p, t, i);
    t.valid[i] = r0 < t.Lq;
    int kv_end = t.Lk;
    if (p.causal) kv_end = min(kv_end, r0 + kTileM);
    t.n[i] = t.valid[i] ? (kv_end + kTileN - 1) / kTileN : 0;
  }
}

// The k-th work tile of this CTA under a static schedule (balanced lists or
// striding); false past the end of its share.
__device__ __forceinline__ bool next_tile(const FwdParams& p, int k, FwdTile& t) {
  int v;
  if (p.tile_list) {
    const int first = __ldg(p.cta_start + blockIdx.x) + k;
    if (first >= __ldg(p.cta_start + blockIdx.x + 1)) return false;
    v = __ldg(p.tile_list + first);
  } else {
    v = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    const int total = p.cu_seqlens ? p.tile_start[p.B] : p.total_tiles;
    if (v >= total) return false;
  }
  expand_fwd_work(p, locate_fwd_work(p, v), t);
  return true;
}

// The k-th work tile of this CTA under a claimed schedule, as the scheduler
// warp published it; false past the end of the work list. `warp_reader` makes lane 0 release the slot
// for the whole warp once every lane has read it (a single-thread reader
// releases it itself). A wait that runs out sets `ok` to false.
__device__ __forceinline__ bool read_tile(FwdBars* bars, int k, FwdTile& t, long long lim,
                                          bool warp_reader, bool& ok) {
  const int slot = k % kSchedSlots;
  // a warp decides together (the broadcast below needs every lane), even when
  // the wait runs out
  const uint32_t full = smem_addr(&bars->sched_full[slot]);
  const uint32_t parity = (k / kSchedSlots) & 1;
  if (!(warp_reader ? mbar_wait_warp(full, parity, lim) : mbar_wait(full, parity, lim))) {
    ok = false;
    return false;
  }
  const int4* src = reinterpret_cast<const int4*>(&bars->sched_t[slot]);
  int4* dst = reinterpret_cast<int4*>(&t);
#pragma unroll
  for (int w = 0; w < static_cast<int>(sizeof(FwdTile) / 16); ++w) dst[w] = src[w];
  if (warp_reader) {
    // lane 0's copy, broadcast, so the compiler knows every field is the same
    // in all lanes (warp-uniform loop bounds and addresses)
    int* f = reinterpret_cast<int*>(&t);
#pragma unroll
    for (int w = 0; w < static_cast<int>(sizeof(FwdTile) / 4); ++w)
      f[w] = __shfl_sync(0xffffffffu, f[w], 0);
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&bars->sched_empty[slot]));
  } else {
    mbar_arrive(smem_addr(&bars->sched_empty[slot]));
  }
  return t.b >= 0;
}

template <int DQK, int DV, int EMU, bool CLAIMED>
__global__ void __launch_bounds__(384, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const FwdParams p) {
  using Cfg = FwdCfg<DQK, DV>;
  // The staged O epilogue pays at d = 64 and for packed inputs (short work
  // tiles, where the epilogue weighs most); with d = 128 and fixed lengths the
  // tiles are long and direct row stores measured faster.
  constexpr bool kTmaEpiUsed = Cfg::kTmaEpi && (DQK == 64 || CLAIMED);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + Cfg::kBarOff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    mbar_init(smem_addr(&bars->q_full), 1);
    mbar_init(smem_addr(&bars->q_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&bars->s_full[i]), 1);
      mbar_init(smem_addr(&bars->p_part[i]), 128);
      mbar_init(smem_addr(&bars->p_full[i]), 128);
      mbar_init(smem_addr(&bars->pv_done[i]), 1);
      mbar_init(smem_addr(&bars->s_free[i]), 128);
    }
    // tile ring: kv_full / kv_empty per stage; block ring: kv_full per load in
    // flight, kv_empty per slot
    for (int i = 0; i < (Cfg::kBlockRing ? Cfg::kSlots : Cfg::kStages); ++i) {
      mbar_init(smem_addr(&bars->kv_full[i]), 1);
      mbar_init(smem_addr(&bars->kv_empty[i]), 1);
    }
    if constexpr (CLAIMED) {
      for (int i = 0; i < kSchedSlots; ++i) {
        mbar_init(smem_addr(&bars->sched_full[i]), 1);
        mbar_init(smem_addr(&bars->sched_empty[i]), kSchedReaders);
      }
    }
    if constexpr (CLAIMED) bars->sched_taken = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&bars->tmem_base), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const long long lim = p.wait_limit;

  // Every role walks the same sequence of work tiles. Barrier phases carry on
  // across tiles, so each role counts its own waits.
  //
  // Register split: 128 x 88 (warps 0-3) + 256 x 208 (softmax) = 384 x 168.
  // Each budget change sits inside the branch of the warps it applies to, so the
  // compiler sees which code runs under which budget.
  if (warp < 4) {
    regs_dec<88>();
  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t ld = 0;   // K/V loads issued so far (K_j, V_j of each tile in turn)
      uint32_t pos = 0;  // block ring: block slots filled so far
      int qk = 0;        // tiles whose Q was loaded (tiles that see no key load nothing)
      FwdTile t;
      bool ok = true;
      for (int k = 0; ok && (CLAIMED ? read_tile(bars, k, t, lim, false, ok) : next_tile(p, k, t)); ++k) {
        if constexpr (CLAIMED) *reinterpret_cast<volatile int*>(&bars->sched_taken) = k + 1;
        const int n_kv = max(t.n[0], t.n[1]);
        if (n_kv > 0) {
          // Q of this tile goes into the buffer once the previous tile's last
          // S MMA has read it
          if (qk > 0 && !mbar_wait(smem_addr(&bars->q_empty), (qk - 1) & 1, lim)) {
            record_error(p.err, kErrTimeout);
            break;
          }
          ++qk;
          const uint32_t qbar = smem_addr(&bars->q_full);
          const int nq = (t.n[0] > 0) + (t.n[1] > 0);
          mbar_arrive_expect_tx(qbar, nq * Cfg::kQTileBytes);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (t.n[i] == 0) continue;
            const uint32_t dst = smem_addr(smem + Cfg::kQOff + i * Cfg::kQTileBytes);
            for (int hf = 0; hf < Cfg::kQBlocks; ++hf)
              tma_load_4d(dst + hf * 16384, &tm_q, qbar, hf * 64, qtile_head(p, t, i),
                          t.row_base + qtile_row(p, t, i), t.batch_coord);
          }
          for (int it = 0; it < 2 * n_kv; ++it, ++ld) {
            const int j = it >> 1;
            const CUtensorMap* map = (it & 1) ? &tm_v : &tm_k;
            if constexpr (!Cfg::kBlockRing) {
              const uint32_t stage = ld % Cfg::kStages;
              const uint32_t round = ld / Cfg::kStages;
              if (!mbar_wait(smem_addr(&bars->kv_empty[stage]), (round & 1) ^ 1, lim)) {
                record_error(p.err, kErrTimeout);
                ok = false;
                break;
              }
              const uint32_t fbar = smem_addr(&bars->kv_full[stage]);
              mbar_arrive_expect_tx(fbar, Cfg::kTileBytes);
              const uint32_t dst = smem_addr(smem + Cfg::kKVOff + stage * Cfg::kTileBytes);
              for (int hf = 0; hf < Cfg::kQBlocks; ++hf)
                tma_load_4d(dst + hf * 16384, map, fbar, hf * 64, t.h_kv, t.row_base + j * kTileN,
                            t.batch_coord);
            } else {
              // block ring: the load's blocks go to slots pos, pos + 1, ... (mod 8).
              // V is read as an MN-major operand whose two column blocks must be
              // a fixed stride apart; when it wraps (slots 7 and 0) its first
              // column block goes to slot 0 and its second to slot 7.
              const int nb = (it & 1) ? Cfg::kVBlocks : Cfg::kQBlocks;
              const uint32_t fbar = smem_addr(&bars->kv_full[ld % Cfg::kFullBars]);
              mbar_arrive_expect_tx(fbar, nb * Cfg::kBlockBytes);
              const bool wrap_v = (it & 1) && (pos % Cfg::kSlots) == Cfg::kSlots - 1;
              for (int blk = 0; blk < nb; ++blk, ++pos) {
                const uint32_t slot = pos % Cfg::kSlots;
                if (!mbar_wait(smem_addr(&bars->kv_empty[slot]), ((pos / Cfg::kSlots) & 1) ^ 1,
                               lim)) {
                  record_error(p.err, kErrTimeout);
                  ok = false;
                  break;
                }
                const int col_blk = wrap_v ? (1 - blk) : blk;
                tma_load_4d(smem_addr(smem + Cfg::kKVOff + slot * Cfg::kBlockBytes), map, fbar,
                            col_blk * 64, t.h_kv, t.row_base + j * kTileN, t.batch_coord);
              }
              if (!ok) break;
            }
          }
        }
      }
      if (!ok) record_error(p.err, kErrTimeout);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the issue loop (so descriptors, phases and tile
    // fields are warp-uniform values) and one elected lane issues each MMA and
    // commit. The issue order alternates the two query tiles (PV_0, S_0, PV_1,
    // S_1, ...), which keeps the two softmax warpgroups half an iteration apart,
    // so each one's softmax overlaps the other tile's MMAs. A tcgen05.mma holds
    // the issuing lane for about its own execution time, so the loop does as
    // little else as possible between MMAs.
    {
      const bool leader = elect_one_sync();
      constexpr uint32_t kIdS = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t kIdPV = make_idesc_bf16(128, DV, 0, 1);
      constexpr int kQB = Cfg::kQBlocks, kVB = Cfg::kVBlocks;
      const uint32_t q_base = smem_addr(smem + Cfg::kQOff);
      const uint32_t kv_base = smem_addr(smem + Cfg::kKVOff);
      // Descriptors are built once; each MMA only adds a byte offset (>> 4) to
      // the start-address field (compile-time for the tile ring).
      const uint64_t q_desc = make_sdesc_sw128(q_base, 16, 1024);     // K-major
      const uint64_t k_desc = make_sdesc_sw128(kv_base, 16, 1024);    // K-major
      const uint64_t v_desc = make_sdesc_sw128(kv_base, 16384, 1024); // MN-major
      // block ring, V wrapped over the ring's end: first column block in slot 0,
      // second in slot 7
      const uint64_t v_desc_wrap = make_sdesc_sw128(kv_base, 7 * 16384, 1024);
      uint32_t ld = 0;     // K/V loads consumed so far, in the producer's order
      uint32_t pos = 0;    // block ring: block slots consumed so far
      // Load `it` of the current tile (K_j = 2j, V_j = 2j + 1): its barrier, its
      // phase, its place in shared memory.
      auto stage_of = [&](int it) { return (ld + it) % Cfg::kStages; };
      auto pos_of = [&](int it) { return pos + (it >> 1) * (kQB + kVB) + ((it & 1) ? kQB : 0); };
      auto full_bar = [&](int it) {
        if constexpr (Cfg::kBlockRing) return smem_addr(&bars->kv_full[(ld + it) % Cfg::kFullBars]);
        else return smem_addr(&bars->kv_full[stage_of(it)]);
      };
      auto full_phase = [&](int it) -> uint32_t {
        if constexpr (Cfg::kBlockRing) return ((ld + it) / Cfg::kFullBars) & 1;
        else return ((ld + it) / Cfg::kStages) & 1;
      };
      auto release = [&](int it) {  // the load's buffer is free once the MMAs so far are done
        if constexpr (Cfg::kBlockRing) {
          const uint32_t p0 = pos_of(it);
          const int nb = (it & 1) ? kVB : kQB;
          for (int b = 0; b < nb; ++b) mma_commit_by(leader, smem_addr(&bars->kv_empty[(p0 + b) % Cfg::kSlots]));
        } else {
          mma_commit_by(leader, smem_addr(&bars->kv_empty[stage_of(it)]));
        }
      };
      auto issue_s = [&](int i, int it) {
        uint64_t qa = q_desc + ((i * Cfg::kQTileBytes) >> 4);
        // With 12 K steps per S the compiler would keep every Q descriptor of
        // both tiles live across the loop and spill; an opaque copy makes it
        // add the offsets at each issue instead.
        if constexpr (Cfg::kBlockRing) asm volatile("" : "+l"(qa));
        const uint32_t d_tmem = tmem + Cfg::kColS0 + i * 128;
        if constexpr (Cfg::kBlockRing) {
          const uint32_t p0 = pos_of(it);
#pragma unroll
          for (int b = 0; b < kQB; ++b) {
            const uint64_t kb = k_desc + ((((p0 + b) % Cfg::kSlots) * 16384) >> 4);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int kk = 4 * b + k4;
              const uint32_t qoff = (b * 16384 + k4 * 32) >> 4;
              mma_ss_by(leader, d_tmem, qa + qoff, kb + ((k4 * 32) >> 4), kIdS, kk > 0);
            }
          }
        } else {
          const uint64_t kb = k_desc + ((stage_of(it) * Cfg::kTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            mma_ss_by(leader, d_tmem, qa + off, kb + off, kIdS, kk > 0);
          }
        }
        mma_commit_by(leader, smem_addr(&bars->s_full[i]));
      };
      // O_i += P_i V_j over the K-steps [K0, K1) (16 keys each)
      auto issue_pv = [&](int i, int it, bool acc, auto k0_, auto k1_) {
        constexpr int K0 = decltype(k0_)::value, K1 = decltype(k1_)::value;
        uint64_t vb;
        if constexpr (Cfg::kBlockRing) {
          const uint32_t slot = pos_of(it) % Cfg::kSlots;
          vb = (slot == Cfg::kSlots - 1) ? v_desc_wrap : v_desc + ((slot * 16384) >> 4);
        } else {
          vb = v_desc + ((stage_of(it) * Cfg::kTileBytes) >> 4);
        }
        const uint32_t d_tmem = tmem + Cfg::kColO0 + i * DV;
        const uint32_t a_tmem = tmem + Cfg::kColP0 + i * Cfg::kColPStep;
#pragma unroll
        for (int kk = K0; kk < K1; ++kk)
          mma_ts_by(leader, d_tmem, a_tmem + kk * 8, vb + kk * (2048 >> 4), kIdPV, (acc || kk > 0));
      };
      using KAll0 = std::integral_constant<int, 0>;
      using KPart = std::integral_constant<int, kPvSteps0>;
      using KAll1 = std::integral_constant<int, kTileN / 16>;
      int pw[2] = {0, 0};  // p_full waits so far, per query tile
      int qk = 0;          // tiles with a Q load
      bool ok = true;
      FwdTile t;
      if constexpr (Cfg::kSepP) {
        // P in its own TMEM columns: S_i of key tile j + 1 is issued once the
        // softmax warpgroup has S_i(j) in registers (s_free), before P_i(j) is
        // ready, so the tensor core computes the next scores while the
        // softmax runs (the order of the four MMAs of a key tile depends on
        // the mask, below), and every PV is committed to pv_done (the softmax
        // waits for PV_i(j) before it writes P_i(j+1) into the same columns).
        int sf[2] = {0, 0};  // s_free waits so far, per query tile
        int ns[2] = {0, 0};  // S MMAs issued so far, per query tile
        auto wait_free_issue_s = [&](int i, int it) {
          if (ns[i] > 0) {  // the softmax has read the previous S_i
            if (!mbar_wait_warp(smem_addr(&bars->s_free[i]), sf[i] & 1, lim)) return false;
            ++sf[i];
            tc_fence_after();
          }
          issue_s(i, it);
          ++ns[i];
          return true;
        };
        for (int k = 0; ok && (CLAIMED ? read_tile(bars, k, t, lim, true, ok) : next_tile(p, k, t)); ++k) {
          const int n_kv = max(t.n[0], t.n[1]);
          if (n_kv == 0) continue;  // no keys: the epilogue writes O = 0, LSE = -inf
          ok = mbar_wait_warp(smem_addr(&bars->q_full), qk & 1, lim);
          ++qk;
          if (ok) ok = mbar_wait_warp(full_bar(0), full_phase(0), lim);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int i = 0; i < 2; ++i)
            if (ok && t.n[i] > 0) ok = wait_free_issue_s(i, 0);
          if (!ok) break;
          release(0);
          if (n_kv == 1) mma_commit_by(leader, smem_addr(&bars->q_empty));
          for (int j = 0; j < n_kv; ++j) {
            const int itv = 2 * j + 1, itk = 2 * j + 2;
            const bool next_k = j + 1 < n_kv;
            if (next_k && !(ok = mbar_wait_warp(full_bar(itk), full_phase(itk), lim))) break;
            if (!(ok = mbar_wait_warp(full_bar(itv), full_phase(itv), lim))) break;
            auto s_next = [&](int i) {  // S_i(j+1), once the softmax has S_i(j)
              if (ok && j + 1 < t.n[i]) ok = wait_free_issue_s(i, itk);
            };
            auto pv_now = [&](int i) {  // O_i += P_i(j) V_j
              if (!ok || j >= t.n[i]) return;
              if (!(ok = mbar_wait_warp(smem_addr(&bars->p_full[i]), pw[i] & 1, lim))) return;
              ++pw[i];
              tc_fence_after();
              issue_pv(i, itv, j > 0, KAll0{}, KAll1{});
              mma_commit_by(leader, smem_addr(&bars->pv_done[i]));
            };
            if (p.causal) {
              // S_0(j+1), S_1(j+1), PV_0(j), PV_1(j): the two query tiles of a
              // causal work tile see different key counts and masks, which
              // already keeps their softmax warpgroups apart
              s_next(0); s_next(1); pv_now(0); pv_now(1);
            } else {
              // S_0(j+1), PV_0(j), S_1(j+1), PV_1(j): query tile 1's S waits
              // behind query tile 0's PV, which staggers two equal query
              // tiles by about one PV + S instead of letting their softmax
              // warpgroups run in lockstep and compete for issue slots
              s_next(0); pv_now(0); s_next(1); pv_now(1);
            }
            if (!ok) break;
            if (next_k) release(itk);  // after the last S reading K_{j+1}
            release(itv);              // after the last PV reading V_j
            // Q is free again once the tile's last S MMA is done
            if (j + 2 == n_kv) mma_commit_by(leader, smem_addr(&bars->q_empty));
          }
          ld += 2 * n_kv;
        }
      } else
      for (int k = 0; ok && (CLAIMED ? read_tile(bars, k, t, lim, true, ok) : next_tile(p, k, t)); ++k) {
        const int n_kv = max(t.n[0], t.n[1]);
        if (n_kv == 0) continue;  // no keys: the epilogue writes O = 0, LSE = -inf
        ok = mbar_wait_warp(smem_addr(&bars->q_full), qk & 1, lim);
        ++qk;
        if (ok) ok = mbar_wait_warp(full_bar(0), full_phase(0), lim);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (t.n[i] > 0) issue_s(i, 0);
        release(0);
        // Q is free again once the tile's last S MMA is done
        if (n_kv == 1) mma_commit_by(leader, smem_addr(&bars->q_empty));
        for (int j = 0; j < n_kv; ++j) {
          const int itv = 2 * j + 1, itk = 2 * j + 2;
          const bool next_k = (j + 1) < n_kv;
          // Block ring (shallow: about 1.6 key/value steps fit): K_{j+1} is waited
          // for only before the first S MMA that reads it, and V_j's slots are
          // released right after its last PV MMA, which gives the producer the
          // earliest start on the following loads.
          bool k_ready = !Cfg::kBlockRing || !next_k;
          ok = mbar_wait_warp(full_bar(itv), full_phase(itv), lim);
          if (ok && next_k && !Cfg::kBlockRing) ok = mbar_wait_warp(full_bar(itk), full_phase(itk), lim);
          if (!ok) break;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (j >= t.n[i]) continue;
            if constexpr (kPvSteps0 < kTileN / 16) {
              // the first three quarters of P_i, then the rest
              if (!mbar_wait_warp(smem_addr(&bars->p_part[i]), pw[i] & 1, lim)) { ok = false; break; }
              tc_fence_after();
              issue_pv(i, itv, j > 0, KAll0{}, KPart{});
              if (!mbar_wait_warp(smem_addr(&bars->p_full[i]), pw[i] & 1, lim)) { ok = false; break; }
              tc_fence_after();
              issue_pv(i, itv, true, KPart{}, KAll1{});
            } else {
              if (!mbar_wait_warp(smem_addr(&bars->p_full[i]), pw[i] & 1, lim)) { ok = false; break; }
              tc_fence_after();
              issue_pv(i, itv, j > 0, KAll0{}, KAll1{});
            }
            ++pw[i];
            if constexpr (Cfg::kBlockRing) {
              if (i == 1 || j >= t.n[1]) release(itv);  // the last PV reading V_j
            }
            // only the last PV of a tile is signalled (to the epilogue); earlier
            // ones are covered by the commit of the S MMA issued after them
            if (j + 1 == t.n[i]) {
              mma_commit_by(leader, smem_addr(&bars->pv_done[i]));
            } else {
              if (!k_ready) {
                if (!(ok = mbar_wait_warp(full_bar(itk), full_phase(itk), lim))) break;
                k_ready = true;
              }
              issue_s(i, itk);
            }
          }
          if (!ok) break;
          if (!Cfg::kBlockRing) release(itv);
          if (next_k) release(itk);
          if (j + 2 == n_kv) mma_commit_by(leader, smem_addr(&bars->q_empty));
        }
        ld += 2 * n_kv;
        pos += n_kv * (kQB + kVB);
      }
      if (!ok && leader) record_error(p.err, kErrTimeout);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- scheduler
    // Claimed schedule (CLAIMED, tile_ctr set): the CTA starts with work tile
    // blockIdx.x and claims every further one from a counter in global memory
    // (zeroed before the launch), so CTAs that finish early take more tiles:
    // greedy list scheduling over the longest-first work list. This warp
    // decodes each claimed tile and hands it to the other roles through a ring
    // of kSchedSlots slots. Under a static schedule the warp is idle and every
    // role decodes its tiles itself.
    if (CLAIMED && lane == 0) {
      const int total = p.cu_seqlens ? p.tile_start[p.B] : p.total_tiles;
      // the sequence of the last decoded tile, kept: consecutive claims of a
      // CTA mostly fall in the same sequence
      int c_t0 = 1, c_t1 = 0;  // its tile range [c_t0, c_t1) (empty: none kept)
      FwdWork c_w;
      c_w.b = 0; c_w.row_base = 0; c_w.L = 0; c_w.local = 0;
      auto locate = [&](int v) {
        if (p.cu_seqlens == nullptr) return locate_fwd_work(p, v);
        if (v < c_t0 || v >= c_t1) {
          // largest virtual sequence whose first tile is <= v
          int lo = 0, hi = p.B;
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.tile_start[mid] <= v) lo = mid; else hi = mid;
          }
          c_t0 = p.tile_start[lo];
          c_t1 = p.tile_start[lo + 1];
          c_w.b = p.seq_order[lo];
          const SeqSpan sp = seq_span(p.cu_seqlens, c_w.b, p.N_q, 0);
          c_w.row_base = sp.start;
          c_w.L = sp.len;
        }
        FwdWork w = c_w;
        w.local = v - c_t0;
        return w;
      };
      // Far from the end of the work list the next tile is claimed as soon as
      // the last one is handed out, so the other roles never wait for a
      // claim. In the last kNearRounds rounds a tile is claimed only once the
      // producer has taken the one before, so no CTA holds large claimed tiles
      // while others run out of work.
      constexpr unsigned kNearRounds = 4;
      bool near_end = false;
      auto claim = [&](int k) {
        unsigned u = blockIdx.x;
        if (k > 0) {
          const unsigned c = atomicAdd(reinterpret_cast<unsigned*>(p.tile_ctr), 1u);
          u = c >= static_cast<unsigned>(total) ? total : gridDim.x + c;
        }
        near_end = u + kNearRounds * gridDim.x >= static_cast<unsigned>(total);
        FwdTile t;
        if (u < static_cast<unsigned>(total)) {
          expand_fwd_work(p, locate(static_cast<int>(u)), t);
        } else {
          t = FwdTile{};
          t.b = -1;
        }
        return t;
      };
      FwdTile t = claim(0);
      for (int k = 0;; ++k) {
        const int slot = k % kSchedSlots;
        if (k >= kSchedSlots && !mbar_wait_sleep(smem_addr(&bars->sched_empty[slot]),
                                                 ((k / kSchedSlots) - 1) & 1, lim, 200)) {
          record_error(p.err, kErrTimeout);
          break;
        }
        bars->sched_t[slot] = t;
        mbar_arrive(smem_addr(&bars->sched_full[slot]));
        if (t.b < 0) break;
        if (near_end) {
          // the producer has taken tile k (a plain counter it raises; no data
          // depends on it)
          bool taken = *reinterpret_cast<volatile int*>(&bars->sched_taken) > k;
          const long long t0 = clock64();
          while (!taken) {
            if (clock64() - t0 > lim) break;
            __nanosleep(100);
            taken = *reinterpret_cast<volatile int*>(&bars->sched_taken) > k;
          }
          if (!taken) {  // the other roles' bounded waits end the CTA
            record_error(p.err, kErrTimeout);
            break;
          }
        }
        t = claim(k + 1);
      }
    }
  }
    __syncwarp();
  } else {
    regs_inc<208>();
    // ---------------------------------------------------------- softmax + epilogue
    const int i = (warp - 4) >> 2;          // query tile of this warpgroup
    const int r = tid - 128 * (1 + i);      // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((r & ~31)) << 16;
    const uint32_t col_s = i ? Cfg::kColS1 : Cfg::kColS0;
    const uint32_t col_o = i ? Cfg::kColO1 : Cfg::kColO0;
    const uint32_t col_p = Cfg::kColP0 + i * Cfg::kColPStep;  // P (over S unless kSepP)
    const float c = p.scale_log2;
    int sw = 0;   // s_full waits so far
    int pvw = 0;  // pv_done waits so far
    int pvc = 0;  // separate P: PV MMAs of this query tile in earlier work tiles
    bool ok = true;
    for (int k = 0; ok; ++k) {
      FwdTile t;
      if (!(CLAIMED ? read_tile(bars, k, t, lim, true, ok) : next_tile(p, k, t))) break;
      const int my_n = i ? t.n[1] : t.n[0];
      const int Lk = t.Lk;
      const int q0i = qtile_row(p, t, i);  // first row of this warpgroup's query tile
      const int qrow = q0i + r;            // sequence-relative query row
      float m_used = -INFINITY;
      float l = 0.0f;
      for (int j = 0; j < my_n; ++j) {
        if (!mbar_wait(smem_addr(&bars->s_full[i]), sw & 1, lim)) { ok = false; break; }
        ++sw;
        tc_fence_after();
        float s[128];
        {
          uint32_t* sr = reinterpret_cast<uint32_t*>(s);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            tmem_ld32(tmem + lane_base + col_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + cc * 32));
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sr + cc * 32));
        }
        if constexpr (Cfg::kSepP) {
          // S_i(j) is in registers: the MMA warp may write S_i(j + 1) now
          tc_fence_before();
          mbar_arrive(smem_addr(&bars->s_free[i]));
        }
        const int kv0 = j * kTileN;
        const bool need_mask = (kv0 + kTileN > Lk) || (p.causal && kv0 + kTileN - 1 > q0i);
        uint32_t pk[64];
        bool rescale_warp;
        float factor;
        const bool pos = c > 0.0f;
        const float mb =
            pos ? softmax_row_max<true>(s, c, m_used, l, kv0, qrow, Lk, need_mask, p.causal,
                                        rescale_warp, factor)
                : softmax_row_max<false>(s, c, m_used, l, kv0, qrow, Lk, need_mask, p.causal,
                                         rescale_warp, factor);
#if ATTN_COUNT_RESCALE
        if (j > 0) {
          const unsigned moved = __ballot_sync(0xffffffffu, rescale_warp && factor != 1.0f);
          if ((r & 31) == 0) {
            atomicAdd(&g_rescale_stats[0], 1ull);
            if (moved) atomicAdd(&g_rescale_stats[1], 1ull);
            atomicAdd(&g_rescale_stats[2], static_cast<unsigned long long>(__popc(moved)));
            atomicAdd(&g_rescale_stats[3], 32ull);
          }
        }
#endif
        uint64_t sum2[2] = {0ull, 0ull};
        if (pos) softmax_row_exp<EMU, true, 0, kPWords0>(s, c, mb, need_mask, pk, sum2);
        else softmax_row_exp<0, false, 0, kPWords0>(s, c, mb, need_mask, pk, sum2);
        if (Cfg::kSepP && j > 0) {
          // PV_i(j - 1) has read P_i(j - 1) and finished O_{j-1}. Waiting on its
          // own phase is unambiguous: S_i(j) completed, and it was issued after
          // PV_i(j - 2), so at most this one PV is outstanding.
          if (!mbar_wait(smem_addr(&bars->pv_done[i]), (pvc + j - 1) & 1, lim)) { ok = false; break; }
          tc_fence_after();
        }
        if (rescale_warp && j > 0 && __any_sync(0xffffffffu, factor != 1.0f)) {
          // correction: O_{j-1} is complete here (P over S: the commit that
          // signalled S_j came from the thread that issued PV_{j-1} before S_j;
          // separate P: the wait above); it is back in TMEM before the first
          // part of P is signalled, so before PV_j adds to O
#pragma unroll
          for (int cc = 0; cc < DV / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_base + col_o + cc * 32, ov);
            tmem_ld_wait(ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
            tmem_st32(tmem + lane_base + col_o + cc * 32, ov);
          }
        }
        tmem_st32(tmem + lane_base + col_p, *reinterpret_cast<uint32_t(*)[32]>(pk));
        if constexpr (kPWords0 < 64 && !Cfg::kSepP) {
          tmem_st16(tmem + lane_base + col_s + 32, *reinterpret_cast<uint32_t(*)[16]>(pk + 32));
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(smem_addr(&bars->p_part[i]));
          if (pos) softmax_row_exp<EMU, true, kPWords0, 64>(s, c, mb, need_mask, pk, sum2);
          else softmax_row_exp<0, false, kPWords0, 64>(s, c, mb, need_mask, pk, sum2);
          tmem_st16(tmem + lane_base + col_s + 48, *reinterpret_cast<uint32_t(*)[16]>(pk + 48));
        } else {
          tmem_st32(tmem + lane_base + col_p + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_addr(&bars->p_full[i]));
        l += softmax_row_sum(sum2);
      }
      if (!ok) break;
      // -------------------------------------------------------- epilogue
      // The O columns are reused by the next tile's first PV MMA, which waits
      // for this warpgroup's next p_full arrival, i.e. after these loads.
      if (i ? t.valid[1] : t.valid[0]) {
        bool have_o = my_n > 0;
        if (have_o) {
          // the tile's last PV (separate P: every PV is committed, so the
          // phase is that PV's own)
          have_o = mbar_wait(smem_addr(&bars->pv_done[i]),
                             Cfg::kSepP ? (pvc + my_n - 1) & 1 : pvw & 1, lim);
          ++pvw;
          if (!have_o) { ok = false; break; }
          tc_fence_after();
        }
        const bool row_ok = qrow < t.Lq;
        const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
        const size_t grow = static_cast<size_t>(t.row_base) + qrow;  // packed row
        const int hq = qtile_head(p, t, i);
        const size_t o_off =
            p.cu_seqlens ? (grow * p.H_q + hq) * DV
                         : ((static_cast<size_t>(t.b) * p.N_q + qrow) * p.H_q + hq) * DV;
        uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + o_off);
        // the row's O columns are loaded with every load in flight at once (one
        // wait instead of one per 32 columns), then scaled, rounded and stored
        // (the last tile of a packed sequence row by row: a 128-row box would
        // also write the next sequence's rows)
        const bool tma_epi = kTmaEpiUsed && (p.cu_seqlens == nullptr || q0i + kTileM <= t.Lq);
        uint32_t ov[DV];
        if (have_o) {
#pragma unroll
          for (int cc = 0; cc < DV / 32; ++cc)
            tmem_ld32(tmem + lane_base + col_o + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(ov + cc * 32));
#pragma unroll
          for (int cc = 0; cc < DV / 32; ++cc) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(ov + cc * 32));
        } else {
#pragma unroll
          for (int e = 0; e < DV; ++e) ov[e] = 0u;
        }
        if (tma_epi) {
          // 64 columns at a time into this warpgroup's swizzled staging buffer,
          // then one TMA store of the 128 x 64 box; the buffer is refilled once
          // the previous store has read it
          uint32_t buf_off = Cfg::kOEpiOff + i * Cfg::kBlockBytes;
          asm volatile("" : "+r"(buf_off));  // computed here, not kept across the key loop
          uint8_t* buf = smem + buf_off;
#pragma unroll
          for (int hf = 0; hf < DV / 64; ++hf) {
            uint32_t w[32];  // scaled and rounded before the wait, so the fp32 values can go
#pragma unroll
            for (int e = 0; e < 32; ++e)
              w[e] = pack_bf16x2(__uint_as_float(ov[hf * 64 + 2 * e]) * inv_l,
                                 __uint_as_float(ov[hf * 64 + 2 * e + 1]) * inv_l);
            if (r == 0) bulk_wait_group_read<0>();
            named_bar_sync(2 + i, 128);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(buf + sw128_offset(r, ch)) =
                  make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
            fence_async_shared();
            named_bar_sync(2 + i, 128);
            if (r == 0) {
              tma_store_4d(&tm_o, smem_addr(buf), hf * 64, hq, t.row_base + q0i, t.batch_coord);
              bulk_commit_group();
            }
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < DV / 32; ++cc) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack_bf16x2(__uint_as_float(ov[cc * 32 + 2 * e]) * inv_l,
                                 __uint_as_float(ov[cc * 32 + 2 * e + 1]) * inv_l);
            if (row_ok) {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                orow[cc * 4 + e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
            }
          }
        }
        if (row_ok) {
          const float lse = (l > 0.0f) ? (m_used * kLn2 + __logf(l)) : -INFINITY;
          const size_t l_off = p.cu_seqlens
                                   ? static_cast<size_t>(hq) * p.N_q + grow
                                   : (static_cast<size_t>(t.b) * p.H_q + hq) * p.N_q + qrow;
          p.lse[l_off] = lse;
        }
      }
      pvc += my_n;
    }
    // the O stores have read the staging buffer before the CTA's shared memory goes
    if (kTmaEpiUsed && r == 0) bulk_wait_group<0>();
    if (!ok) record_error(p.err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// Orders packed sequences longest first (their longest work item is the
// longest) and writes a work list's metadata: seq_order maps a virtual
// sequence index to the actual one and tile_start[v] is the first work item of
// virtual sequence v, a sequence of L rows having ceil(L / rows) * units items
// (FlashAttention-4 summary, section 3.3, the varlen scheduling paragraph).
// The forward's items are its work tiles, the backward's its (key tile, KV
// head) items. One CTA. Ties keep their input order; with sort == 0 the input
// order is kept.
__global__ void __launch_bounds__(1024)
seq_plan_kernel(const int* __restrict__ cu_seqlens, int B, int T, int rows, int units, int sort,
                int* seq_order, int* tile_start, int* tile_ctr, int* err) {
  extern __shared__ int plan_smem[];
  int* len = plan_smem;        // [B] when sorting
  int* ord = plan_smem + B;    // [B] when sorting
  __shared__ int warp_sum[32];
  const int tid = threadIdx.x;
  if (tid == 0 && tile_ctr != nullptr) *tile_ctr = 0;  // the forward's claim counter
  // the lengths are those the kernels decode (clamped into the T packed rows);
  // an inconsistent offset array is reported through the error word
  check_cu_seqlens(cu_seqlens, B, T, err, tid, blockDim.x);
  if (sort) {
    for (int s = tid; s < B; s += blockDim.x) len[s] = seq_span(cu_seqlens, s, T, 0).len;
    __syncthreads();
    for (int s = tid; s < B; s += blockDim.x) {
      const int L = len[s];
      int rank = 0;
      for (int u = 0; u < B; ++u) {
        const int Lu = len[u];
        rank += (Lu > L) || (Lu == L && u < s);
      }
      ord[rank] = s;
    }
    __syncthreads();
  }
  // exclusive prefix of the work tiles per virtual sequence: each thread owns a
  // contiguous chunk, chunk sums are scanned across the block
  const int chunk = (B + blockDim.x - 1) / blockDim.x;
  const int v0 = min(B, tid * chunk), v1 = min(B, v0 + chunk);
  auto tiles_of = [&](int vs) {
    const int s = sort ? ord[vs] : vs;
    const int L = sort ? len[s] : seq_span(cu_seqlens, s, T, 0).len;
    return (L + rows - 1) / rows * units;
  };
  int local = 0;
  for (int vs = v0; vs < v1; ++vs) local += tiles_of(vs);
  const int lane = tid & 31, w = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    int x = lane < nw ? warp_sum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < nw) warp_sum[lane] = x;  // inclusive over warps
  }
  __syncthreads();
  int run = incl - local + (w > 0 ? warp_sum[w - 1] : 0);
  for (int vs = v0; vs < v1; ++vs) {
    seq_order[vs] = sort ? ord[vs] : vs;
    tile_start[vs] = run;
    run += tiles_of(vs);
  }
  if (tid == blockDim.x - 1) tile_start[B] = warp_sum[(blockDim.x >> 5) - 1];
}

// ------------------------------------------------------------------ host side

template <int DQK, int DV, int EMU, bool CLAIMED>
static cudaError_t launch_fwd_impl_sched(const CUtensorMap& tq, const CUtensorMap& tk,
                                         const CUtensorMap& tv, const CUtensorMap& to,
                                         const FwdParams& p, dim3 grid, cudaStream_t stream) {
  using Cfg = FwdCfg<DQK, DV>;
  auto kern = attn_fwd_kernel<DQK, DV, EMU, CLAIMED>;
  constexpr int kSmem = (Cfg::kTmaEpi && (DQK == 64 || CLAIMED)) ? Cfg::kSmemBytesEpi : Cfg::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  static_assert(sizeof(FwdBars) <= 512, "barrier block overflows its reservation");
  const int slot = prof_begin(kKFwd, stream);
  kern<<<grid, 384, kSmem, stream>>>(tq, tk, tv, to, p);
  e = cudaGetLastError();
  prof_end(slot, stream);
  return e;
}

// A claimed schedule (tile_ctr set) runs the instance with the scheduler warp.
template <int DQK, int DV, int EMU>
static cudaError_t launch_fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& to,
                                   const FwdParams& p, dim3 grid, cudaStream_t stream) {
  if (p.tile_ctr != nullptr)
    return launch_fwd_impl_sched<DQK, DV, EMU, true>(tq, tk, tv, to, p, grid, stream);
  return launch_fwd_impl_sched<DQK, DV, EMU, false>(tq, tk, tv, to, p, grid, stream);
}

// Number of exponentials per 8 pairs routed to the FMA polynomial (d = 64 has
// its own setting).
#ifndef ATTN_FWD_EMU
#define ATTN_FWD_EMU 0
#endif
#ifndef ATTN_FWD_EMU_64
#define ATTN_FWD_EMU_64 ATTN_FWD_EMU
#endif

// Supported (d_qk, d_v): (64, 64), (128, 128), (192, 128); the caller checks.
// `to` maps O like `tq` maps Q (d_v columns, 128 x 64 boxes, 128-byte swizzle).
cudaError_t launch_attn_fwd(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p,
                            dim3 grid, cudaStream_t stream) {
  if (d_qk == 64 && d_v == 64)
    return launch_fwd_impl<64, 64, ATTN_FWD_EMU_64>(tq, tk, tv, to, p, grid, stream);
  if (d_qk == 192 && d_v == 128)
    return launch_fwd_impl<192, 128, ATTN_FWD_EMU>(tq, tk, tv, to, p, grid, stream);
  return launch_fwd_impl<128, 128, ATTN_FWD_EMU>(tq, tk, tv, to, p, grid, stream);
}

// Largest packed batch the plan kernel sorts (its lengths and order sit in
// shared memory); larger batches keep their input order.
constexpr int kPlanMaxSort = 8192;

cudaError_t launch_seq_plan(const int* cu_seqlens, int B, int T, int rows, int units,
                            int* seq_order, int* tile_start, int* tile_ctr, int* err, int prof_id,
                            cudaStream_t stream) {
  const int sort = (B <= kPlanMaxSort) ? 1 : 0;
  const size_t smem = sort ? static_cast<size_t>(2) * B * sizeof(int) : 0;
  cudaError_t e = cudaFuncSetAttribute(seq_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       2 * kPlanMaxSort * static_cast<int>(sizeof(int)));
  if (e != cudaSuccess) return e;
  const int slot = prof_begin(prof_id, stream);
  seq_plan_kernel<<<1, 1024, smem, stream>>>(cu_seqlens, B, T, rows, units, sort, seq_order,
                                              tile_start, tile_ctr, err);
  e = cudaGetLastError();
  prof_end(slot, stream);
  return e;
}

cudaError_t launch_fwd_plan(const int* cu_seqlens, int B, int T, int H_q, int pair_heads,
                            int* seq_order, int* tile_start, int* tile_ctr, int* err,
                            cudaStream_t stream) {
  return launch_seq_plan(cu_seqlens, B, T, (2 * kTileM) >> pair_heads, H_q >> pair_heads,
                         seq_order, tile_start, tile_ctr, err, kKFwdPlan, stream);
}

// Reads (and with reset clears) the rescale counters; returns the number of
// values written (0 when the library was built without them).
int read_rescale_stats(unsigned long long* out, int reset) {
#if ATTN_COUNT_RESCALE
  if (cudaMemcpyFromSymbol(out, g_rescale_stats, sizeof(g_rescale_stats)) != cudaSuccess) return -1;
  if (reset) {
    const unsigned long long z[4] = {0ull, 0ull, 0ull, 0ull};
    if (cudaMemcpyToSymbol(g_rescale_stats, z, sizeof(z)) != cudaSuccess) return -1;
  }
  return 4;
#else
  (void)out;
  (void)reset;
  return 0;
#endif
}

// ------------------------------------------------------------------ exp2 test hook
__global__ void exp2_probe_kernel(const float* __restrict__ x, float* __restrict__ y, int n,
                                  int mode) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    if (mode) {
      float y1;
      exp2_poly3_x2(x[i], x[i], y[i], y1);
    } else {
      y[i] = ex2_approx(x[i]);
    }
  }
}

// Failure test: one CTA waits on an mbarrier that nothing ever arrives at. The
// bounded wait gives up after `limit` cycles and records a timeout; nothing
// else is in flight, so the kernel just returns.
__global__ void stall_probe_kernel(int* err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (!mbar_wait(smem_addr(&bar), 0, limit)) {
    if (threadIdx.x == 0) record_error(err, kErrTimeout);
  }
}

cudaError_t launch_stall_probe(int* err, long long limit, cudaStream_t stream) {
  const int slot = prof_begin(kKStall, stream);
  stall_probe_kernel<<<1, 32, 0, stream>>>(err, limit);
  const cudaError_t e = cudaGetLastError();
  prof_end(slot, stream);
  return e;
}

cudaError_t launch_exp2_probe(const float* x, float* y, int n, int mode, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int slot = prof_begin(kKExp2, stream);
  exp2_probe_kernel<<<(n + 255) / 256, 256, 0, stream>>>(x, y, n, mode);
  const cudaError_t e = cudaGetLastError();
  prof_end(slot, stream);
  return e;
}

}  // namespace attn

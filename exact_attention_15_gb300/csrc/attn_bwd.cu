// Backward pass of exact softmax attention for sm_103a: three launches.
//
//   pre   D = rowsum(dO o O) (fp32, laid out like LSE); zero the fp32 dQ
//         accumulator, the ordering semaphores and the work-ticket counter.
//   main  one CTA per key tile j of one (batch, KV head): K_j and V_j stay in
//         shared memory, dK_j and dV_j accumulate in TMEM, and the CTA walks every
//         query tile (of every query head of the GQA group) that sees key tile j.
//         Per query tile i it recomputes P from the saved LSE and issues five
//         tcgen05 contractions (FlashAttention-4 summary, section 3.2.2):
//             S^T  = K Q_i^T        (SS)      P^T = exp2(S^T alpha log2e - LSE_i log2e)
//             dP^T = V dO_i^T       (SS)
//             dV  += P^T dO_i       (TS, P^T from TMEM)
//                                             dS^T = P^T o (dP^T - D_i)
//             dK  += dS^T Q_i       (SS, dS^T from shared memory)
//             dQ_i = dS K           (SS, dS from shared memory)
//         and adds dQ_i into the fp32 accumulator with vector reductions; in
//         deterministic mode the additions into one query tile happen in
//         ascending key-tile order, enforced by a per-tile semaphore
//         (section 3.2.4).
//   post  dQ = alpha * dQacc -> bf16.
//
// Warp roles of the main kernel (512 threads):
//   warp 0      producer: Q_i and dO_i by TMA into a two-stage ring, LSE_i and D_i
//               (plain loads) into the same stage.
//   warp 1      TMEM owner and MMA issuer (one thread).
//   warps 4-11  "compute", two warpgroups: thread r of warpgroup c owns key row r
//               and query columns [64c, 64c+64): P^T, dS^T, and at the end half of
//               the dK / dV row.
//   warps 12-15 "dQ": thread r owns query row r of the dQ_i tile: TMEM -> registers
//               -> fp32 reductions into the accumulator.
//
// TMEM (512 columns): dV [0, d), dK [d, 2d), S^T / P^T [2d, 2d+128),
// dP^T / dQ [2d+128, 2d+256). dS lives only in shared memory: the same
// 128-byte-swizzled buffer is the K-major A operand of dK = dS^T Q and the
// MN-major A operand of dQ = dS K.
#include <cstdint>
#include <cuda_runtime.h>

#include "attn_common.cuh"

namespace attn {

// Shared-memory and TMEM plan of the main kernel. Q and K rows have DQK
// columns, V and dO rows DV; every tile is stored as 128-row x 64-column (16 KB)
// 128-byte-swizzled blocks. A pass computes dK and dQ for the query/key head
// columns [C0, C0 + NC) (all of them when DQK <= 128; DQK = 192 takes two
// passes, 0-127 and 128-191, because dV, dK, S^T and dP^T / dQ of 192 columns
// need 640 of the 512 TMEM columns), and dV in the pass with C0 = 0.
template <int DQK, int DV, int NC>
struct BwdCfg {
  static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= 128 && NC <= 128, "head dimensions");
  static constexpr int kQKBytes = kTileM * DQK * 2;  // one 128-row bf16 tile of Q or K
  static constexpr int kVBytes = kTileM * DV * 2;    // one 128-row bf16 tile of V or dO
  // two Q stages fit next to everything else up to 128 columns; at 192 one
  static constexpr int kQStages = DQK <= 128 ? 2 : 1;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kQKBytes;
  static constexpr int kQOff = kVOff + kVBytes;                 // kQStages stages
  static constexpr int kdOOff = kQOff + kQStages * kQKBytes;    // 1 stage (reloaded once dV is done)
  static constexpr int kdSOff = kdOOff + kVBytes;               // 128 x 128 bf16
  static constexpr int kdQOff = kdSOff + 128 * 128 * 2;         // 2 x (128 rows x 32 fp32) staging
  static constexpr int kStatOff = kdQOff + 2 * 16384;           // per Q stage: lse2[128], D[128]
  static constexpr int kBarOff = kStatOff + kQStages * 2 * 128 * 4;
  static constexpr int kSmemBytes = kBarOff + 256;
  static constexpr uint32_t kColDV = 0, kColDK = DV, kColS = 2 * DV, kColDP = 2 * DV + 128;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColDK + NC <= kColS && kColDP + (NC > 128 ? NC : 128) <= kTmemCols, "TMEM plan");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[2];   // Q_i, LSE_i and D_i of stage i % 2
  uint64_t q_empty[2];
  uint64_t do_full, do_empty;
  uint64_t s_full, dp_full, p_ready, ds_ready, dq_full, dq_free;
  uint32_t tmem_base;
  int work_idx;
};

struct BwdTile {
  int b, h_kv, j;
  int row_base;     // packed-row offset of the sequence (0 fixed length)
  int batch_coord;  // TMA batch coordinate
  int Lq, Lk;
  int i_start, n_qt;  // query tiles [i_start, n_qt) of each query head
  int sem_base;       // first query-tile slot of this sequence (packed) or batch
};

template <bool SPT>
__device__ __forceinline__ bool decode_bwd_tile(const BwdParams& p, int idx, BwdTile& t) {
  if (p.cu_seqlens == nullptr) {
    const int nk = (p.N_k + kTileN - 1) / kTileN;
    if (nk == 0) return false;
    int jj, pair;  // key-tile step and (batch, KV head) pair of the item
    if (p.sec_heads > 0) {
      // causal: sections of sec_heads pairs whose Q and dO fit in L2; inside a
      // section key tile major (every pair's key tile j before key tile j + 1),
      // so the long items near the diagonal's start are dealt out first
      const int per_sec = p.sec_heads * nk;
      const int sec = idx / per_sec;
      const int r = idx - sec * per_sec;
      const int n_pairs = p.B * p.H_kv;
      const int in_sec = min(p.sec_heads, n_pairs - sec * p.sec_heads);
      if (in_sec <= 0) return false;
      jj = r / in_sec;
      pair = sec * p.sec_heads + (r - jj * in_sec);
    } else {
      jj = idx % nk;
      pair = idx / nk;
    }
    t.j = SPT ? nk - 1 - jj : jj;
    t.h_kv = pair % p.H_kv;
    t.b = pair / p.H_kv;
    if (t.b >= p.B) return false;
    t.row_base = 0;
    t.batch_coord = t.b;
    t.Lq = p.N_q;
    t.Lk = p.N_k;
    t.sem_base = t.b * ((p.N_q + kTileM - 1) / kTileM);
  } else if (p.seq_order != nullptr) {
    // sequences longest first; inside one, key tile major (every KV head of key
    // tile j before key tile j + 1), which deals the long items out first
    if (idx >= __ldg(p.item_start + p.B)) return false;
    int lo = 0, hi = p.B;  // largest virtual sequence whose first item is <= idx
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.item_start + mid) <= idx) lo = mid; else hi = mid;
    }
    const int first = __ldg(p.item_start + lo);
    const SeqSpan sp = seq_span(p.cu_seqlens, __ldg(p.seq_order + lo), p.N_q, 0);
    const int L = sp.len;
    const int nk = (L + kTileN - 1) / kTileN;
    const int local = idx - first;
    const int jj = local / p.H_kv;
    t.j = SPT ? nk - 1 - jj : jj;
    t.h_kv = local - jj * p.H_kv;
    t.b = __ldg(p.seq_order + lo);
    t.row_base = sp.start;
    t.batch_coord = 0;
    t.Lq = L;
    t.Lk = L;
    // a sequence's query tiles take the slots after those of the sequences
    // before it in this order; an inconsistent offset array (reported by the
    // planning kernel) could run them past the semaphore array
    t.sem_base = first / p.H_kv;
    if (t.sem_base + (L + kTileM - 1) / kTileM > p.sem_slots) return false;
  } else {
    // sequences in order, each clamped after the one before it (seq_span), so
    // their query-tile slots stay within the semaphore array
    int s = 0, qslots = 0;
    SeqSpan sp{0, 0};
    for (; s < p.B; ++s) {
      sp = seq_span(p.cu_seqlens, s, p.N_q, sp.start + sp.len);
      const int nk = (sp.len + kTileN - 1) / kTileN;
      if (idx < nk * p.H_kv) break;
      idx -= nk * p.H_kv;
      qslots += (sp.len + kTileM - 1) / kTileM;
    }
    if (s >= p.B) return false;
    const int L = sp.len;
    const int nk = (L + kTileN - 1) / kTileN;
    t.j = SPT ? nk - 1 - idx % nk : idx % nk;
    t.h_kv = idx / nk;
    t.b = s;
    t.row_base = sp.start;
    t.batch_coord = 0;
    t.Lq = L;
    t.Lk = L;
    t.sem_base = qslots;
  }
  t.n_qt = (t.Lq + kTileM - 1) / kTileM;
  t.i_start = p.causal ? t.j : 0;
  if (t.i_start > t.n_qt) t.i_start = t.n_qt;
  return true;
}

// Query tile of step k of a key tile's walk (per query head). Deterministic
// order (FlashAttention-4 summary, section 3.2.4): the additions into one dQ
// tile follow a fixed order, and a key tile waits for its turn. With p.spt the
// key tiles start in descending order and the additions into query tile i come
// in walk-step order: under a causal mask a key tile walks up from its diagonal
// (shortest-processing-time first: the first addition of every key tile is the
// first into its query tile); without one, key tile j starts its walk at query
// tile j (same query and key lengths), so at every step each query tile has
// exactly one new contributor. A key tile's k-th addition then waits only for
// additions other key tiles make at their steps before k. Otherwise the walk
// ascends from i_start and the additions come in ascending key-tile order.
// (SPT is a template argument so that the other kernels keep their code.)
template <bool SPT>
__device__ __forceinline__ int bwd_query_tile(const BwdParams& p, const BwdTile& t, int k) {
  if (!SPT || p.causal) return t.i_start + k;
  const int i = t.j + k;
  return i < t.n_qt ? i : i - t.n_qt;
}

// ------------------------------------------------------------------ pre / post

// D[row] = sum_c dO[row, c] * O[row, c] over the D value columns; G = D/16
// lanes per (row, head). Zeroes the fp32 dQ accumulator (n_acc_vec4 float4s)
// and the ints sem[0 .. n_sem].
template <int D>
__global__ void __launch_bounds__(256)
attn_bwd_pre_kernel(const BwdParams p, long long n_rowheads, long long n_acc_vec4, int n_sem) {
  constexpr int G = D / 16;  // lanes per row, 16 elements (32 bytes) each
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  // zero the accumulator and the semaphores
  float4* acc = reinterpret_cast<float4*>(p.dq_acc);
  for (long long i = tid; i < n_acc_vec4; i += nthreads) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.sem != nullptr)  // the semaphores and, after them, the work-ticket counter
    for (long long i = tid; i <= n_sem; i += nthreads) p.sem[i] = 0;
  // an inconsistent packed-sequence offset array is reported (the main kernel
  // clamps what it decodes, so it stays inside the tensors either way)
  if (p.cu_seqlens != nullptr) check_cu_seqlens(p.cu_seqlens, p.B, p.N_q, p.err, tid, nthreads);
  // D: a warp handles 32 / G (row, head) pairs per step; the loop bounds are
  // uniform across the warp so the shuffles below always have every lane.
  const long long warp_id = tid >> 5;
  const long long n_warps = nthreads >> 5;
  const int lane = threadIdx.x & 31;
  const int part = lane % G;
  for (long long w0 = warp_id * (32 / G); w0 < n_rowheads; w0 += n_warps * (32 / G)) {
    const long long rh = w0 + lane / G;  // index into the [rows, H_q] view
    const bool valid = rh < n_rowheads;
    float acc_d = 0.f;
    if (valid) {
      const uint4* o4 = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.o) + rh * D) + part * 2;
      const uint4* g4 = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout) + rh * D) + part * 2;
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const uint4 a = o4[v], g = g4[v];
        const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, gg[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc_d = fmaf(bf16lo_to_f32(aa[e]), bf16lo_to_f32(gg[e]), acc_d);
          acc_d = fmaf(bf16hi_to_f32(aa[e]), bf16hi_to_f32(gg[e]), acc_d);
        }
      }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc_d += __shfl_xor_sync(0xffffffffu, acc_d, off, G);
    if (valid && part == 0) {
      const long long row = rh / p.H_q;
      const int h = static_cast<int>(rh % p.H_q);
      long long idx;
      if (p.cu_seqlens == nullptr) {
        const long long b = row / p.N_q, n = row % p.N_q;
        idx = (b * p.H_q + h) * p.N_q + n;
      } else {
        idx = static_cast<long long>(h) * p.N_q + row;
      }
      p.dvec[idx] = acc_d;
    }
  }
}

__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const BwdParams p, long long n_vec8) {
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_vec8;
       i += nthreads) {
    const float4 a = reinterpret_cast<const float4*>(p.dq_acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(p.dq_acc)[2 * i + 1];
    const float s = p.scale;
    uint4 w;
    w.x = pack_bf16x2(a.x * s, a.y * s);
    w.y = pack_bf16x2(a.z * s, a.w * s);
    w.z = pack_bf16x2(b.x * s, b.y * s);
    w.w = pack_bf16x2(b.z * s, b.w * s);
    reinterpret_cast<uint4*>(p.dq)[i] = w;
  }
}

// ------------------------------------------------------------------ main



template <int DQK, int DV, int C0, int NC, bool SPT>
__global__ void __launch_bounds__(512, 1)
attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv, const BwdParams p, int* ticket) {
  using Cfg = BwdCfg<DQK, DV, NC>;
  constexpr bool kDoDV = C0 == 0;          // this pass also accumulates dV
  constexpr int kQS = Cfg::kQStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + Cfg::kBarOff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if ((smem_addr(smem) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    if (tid == 0) record_error(p.err, kErrTimeout);
    return;
  }
  // Work item: a ticket in deterministic mode (so that every tile a CTA waits
  // on belongs to a CTA that started earlier), the block index otherwise.
  if (tid == 0)
    bars->work_idx = (ticket != nullptr) ? atomicAdd(ticket, 1) : static_cast<int>(blockIdx.x);
  __syncthreads();
  BwdTile t;
  if (!decode_bwd_tile<SPT>(p, bars->work_idx, t)) return;
  const int n_per_head = t.n_qt - t.i_start;
  const int n_it = n_per_head * p.group;
  const long long lim = p.wait_limit;

  if (tid == 0) {
    mbar_init(smem_addr(&bars->kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&bars->q_full[s]), 32);
      mbar_init(smem_addr(&bars->q_empty[s]), 1);
    }
    mbar_init(smem_addr(&bars->do_full), 1);
    mbar_init(smem_addr(&bars->do_empty), 1);
    mbar_init(smem_addr(&bars->s_full), 1);
    mbar_init(smem_addr(&bars->dp_full), 1);
    mbar_init(smem_addr(&bars->p_ready), 256);
    mbar_init(smem_addr(&bars->ds_ready), 256);
    mbar_init(smem_addr(&bars->dq_full), 1);
    mbar_init(smem_addr(&bars->dq_free), 128);
    fence_barrier_init();
    fence_async_shared();
    if (n_it > 0) {
      // K_j, V_j and the first tile's Q and dO go out now (this thread is the
      // producer's lane 0), so their latency overlaps the rest of the set-up
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      const int row_k = t.row_base + t.j * kTileN;
      const uint32_t kvb = smem_addr(&bars->kv_full);
      mbar_arrive_expect_tx(kvb, Cfg::kQKBytes + Cfg::kVBytes);
      for (int hf = 0; hf < DQK / 64; ++hf)
        tma_load_4d(smem_addr(smem + Cfg::kKOff) + hf * 16384, &tm_k, kvb, hf * 64, t.h_kv, row_k,
                    t.batch_coord);
      for (int hf = 0; hf < DV / 64; ++hf)
        tma_load_4d(smem_addr(smem + Cfg::kVOff) + hf * 16384, &tm_v, kvb, hf * 64, t.h_kv, row_k,
                    t.batch_coord);
      const int h0 = t.h_kv * p.group;
      const int row_q = t.row_base + bwd_query_tile<SPT>(p, t, 0) * kTileM;
      const uint32_t fb = smem_addr(&bars->q_full[0]);
      mbar_expect_tx(fb, Cfg::kQKBytes);
      for (int hf = 0; hf < DQK / 64; ++hf)
        tma_load_4d(smem_addr(smem + Cfg::kQOff) + hf * 16384, &tm_q, fb, hf * 64, h0, row_q,
                    t.batch_coord);
      const uint32_t db = smem_addr(&bars->do_full);
      mbar_arrive_expect_tx(db, Cfg::kVBytes);
      for (int hf = 0; hf < DV / 64; ++hf)
        tma_load_4d(smem_addr(smem + Cfg::kdOOff) + hf * 16384, &tm_do, db, hf * 64, h0, row_q,
                    t.batch_coord);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&bars->tmem_base), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // Register split: 128 x 104 (warps 0-3) + 256 x 128 (compute) + 128 x 144 (dQ)
  // = 64,512 <= 512 x 128 (the launch total).
  if (warp < 4) {
    regs_dec<104>();
    if (warp == 0) {
      // ------------------------------------------------------- producer
      if (n_it > 0) {
        // (K_j, V_j and tile 0's Q and dO were issued during the set-up)
        float* stat = reinterpret_cast<float*>(smem + Cfg::kStatOff);
        // LSE (to log2 units) and D of the 128 rows of a query tile, four rows a
        // lane; rows past the end get LSE = +inf so that their P is exactly 0.
        // They are loaded one tile ahead, so the global loads' round trip
        // overlaps the waits for the next Q stage and dO buffer instead of
        // following them.
        float lv[4], dv[4];
        auto load_stats = [&](int it) {
          const int h = t.h_kv * p.group + it / n_per_head;
          const int i = bwd_query_tile<SPT>(p, t, it % n_per_head);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = i * kTileM + lane + 32 * e;
            lv[e] = INFINITY;
            dv[e] = 0.f;
            if (q < t.Lq) {
              const size_t off = p.cu_seqlens
                                     ? static_cast<size_t>(h) * p.N_q + t.row_base + q
                                     : (static_cast<size_t>(t.b) * p.H_q + h) * p.N_q + q;
              lv[e] = p.lse[off];
              dv[e] = p.dvec[off];
            }
          }
        };
        load_stats(0);
        for (int it = 0; it < n_it; ++it) {
          const int stage = it % kQS;
          const int h = t.h_kv * p.group + it / n_per_head;
          const int i = bwd_query_tile<SPT>(p, t, it % n_per_head);
          if (!mbar_wait(smem_addr(&bars->q_empty[stage]), ((it / kQS) & 1) ^ 1, lim)) {
            record_error(p.err, kErrTimeout);
            break;
          }
          const uint32_t fb = smem_addr(&bars->q_full[stage]);
          if (lane == 0 && it > 0) {
            mbar_expect_tx(fb, Cfg::kQKBytes);
            for (int hf = 0; hf < DQK / 64; ++hf)
              tma_load_4d(smem_addr(smem + Cfg::kQOff + stage * Cfg::kQKBytes) + hf * 16384, &tm_q,
                          fb, hf * 64, h, t.row_base + i * kTileM, t.batch_coord);
          }
          float* lse2 = stat + stage * 256;
          float* dvs = lse2 + 128;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float l2 = lv[e] * kLog2e;
            if (l2 == -INFINITY) l2 = INFINITY;  // a row that saw no key has no gradient
            lse2[lane + 32 * e] = l2;
            dvs[lane + 32 * e] = dv[e];
          }
          mbar_arrive(fb);
          if (it + 1 < n_it) load_stats(it + 1);
          // dO_i into the single dO buffer once dV_{i-1} has read it
          if (!mbar_wait(smem_addr(&bars->do_empty), (it & 1) ^ 1, lim)) {
            record_error(p.err, kErrTimeout);
            break;
          }
          if (lane == 0 && it > 0) {
            const uint32_t db = smem_addr(&bars->do_full);
            mbar_arrive_expect_tx(db, Cfg::kVBytes);
            for (int hf = 0; hf < DV / 64; ++hf)
              tma_load_4d(smem_addr(smem + Cfg::kdOOff) + hf * 16384, &tm_do, db, hf * 64, h,
                          t.row_base + i * kTileM, t.batch_coord);
          }
          __syncwarp();
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------- MMA issuer
      // Issue order per query tile i with two Q stages (S_{i+1} goes ahead of
      // dK_i / dQ_i so the tensor core has work while the compute warps turn
      // dP_i into dS_i and S_{i+1} into P_{i+1}):
      //   S_0, dP_0 | dV_i, S_{i+1}, dK_i, dQ_i, dP_{i+1} | ...
      // With one Q stage (DQK = 192) Q_{i+1} can only load once dK_i, the last
      // reader of Q_i, is done:
      //   S_0, dP_0 | dV_i, dK_i, dQ_i, S_{i+1}, dP_{i+1} | ...
      // A pass without dV skips it; dK and dQ cover the pass's NC columns.
      // The whole warp runs the issue loop (warp-uniform descriptors and
      // phases); one elected lane issues each MMA and commit.
      if (n_it > 0) {
        const bool leader = elect_one_sync();
        constexpr uint32_t kIdSS = make_idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
        constexpr uint32_t kIdDV = make_idesc_bf16(128, DV, 0, 1);   // dV: B MN-major
        constexpr uint32_t kIdDK = make_idesc_bf16(128, NC, 0, 1);   // dK: B MN-major
        constexpr uint32_t kIdDQ = make_idesc_bf16(128, NC, 1, 1);   // dQ: A and B MN-major
        // Descriptors are built once; each MMA only adds a compile-time byte
        // offset (>> 4) to the start-address field, which keeps the single
        // issuing thread ahead of the tensor core. Every tile is made of
        // 128-byte-swizzled [rows x 64] blocks that read as K-major (lbo
        // unused) or MN-major (lbo = 16 KB between the 64-column blocks); the
        // pass's columns of Q and K start at block C0 / 64.
        constexpr uint32_t kC0Blk = (C0 / 64) * (16384 >> 4);
        const uint32_t k_base = smem_addr(smem + Cfg::kKOff);
        const uint32_t v_base = smem_addr(smem + Cfg::kVOff);
        const uint32_t ds_base = smem_addr(smem + Cfg::kdSOff);
        const uint64_t k_km = make_sdesc_sw128(k_base, 16, 1024);
        const uint64_t k_mn = make_sdesc_sw128(k_base, 16384, 1024) + kC0Blk;
        const uint64_t v_km = make_sdesc_sw128(v_base, 16, 1024);
        const uint64_t q_km = make_sdesc_sw128(smem_addr(smem + Cfg::kQOff), 16, 1024);
        const uint64_t q_mn = make_sdesc_sw128(smem_addr(smem + Cfg::kQOff), 16384, 1024) + kC0Blk;
        const uint64_t do_km = make_sdesc_sw128(smem_addr(smem + Cfg::kdOOff), 16, 1024);
        const uint64_t do_mn = make_sdesc_sw128(smem_addr(smem + Cfg::kdOOff), 16384, 1024);
        const uint64_t ds_km = make_sdesc_sw128(ds_base, 16, 1024);
        const uint64_t ds_mn = make_sdesc_sw128(ds_base, 16384, 1024);
        constexpr uint32_t kStageStep = Cfg::kQKBytes >> 4;
        auto koff = [](int kk) { return static_cast<uint32_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
        auto issue_s = [&](int it) {  // S^T = K Q^T
          const uint64_t qb = q_km + (it % kQS) * kStageStep;
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            mma_ss_by(leader, tmem + Cfg::kColS, k_km + koff(kk), qb + koff(kk), kIdSS, kk > 0);
          mma_commit_by(leader, smem_addr(&bars->s_full));
        };
        auto issue_dp = [&](int) {  // dP^T = V dO^T
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            mma_ss_by(leader, tmem + Cfg::kColDP, v_km + koff(kk), do_km + koff(kk), kIdSS, kk > 0);
          mma_commit_by(leader, smem_addr(&bars->dp_full));
        };
        auto wait_issue_s = [&](int it) {  // S^T of tile `it` once its Q is in
          if (!mbar_wait_warp(smem_addr(&bars->q_full[it % kQS]), (it / kQS) & 1, lim)) return false;
          tc_fence_after();
          issue_s(it);
          return true;
        };
        bool ok = mbar_wait_warp(smem_addr(&bars->kv_full), 0, lim);
        if (ok) ok = wait_issue_s(0);
        if (ok) ok = mbar_wait_warp(smem_addr(&bars->do_full), 0, lim);
        if (ok) {
          tc_fence_after();
          issue_dp(0);
        }
        for (int it = 0; ok && it < n_it; ++it) {
          const int stage = it % kQS;
          // dV += P^T dO  (P^T from TMEM)
          if (!(ok = mbar_wait_warp(smem_addr(&bars->p_ready), it & 1, lim))) break;
          tc_fence_after();
          if constexpr (kDoDV) {
            // P^T for queries [0, 64) sits in S^T columns [0, 32), for queries
            // [64, 128) in columns [64, 96); each MMA reads one 16-query slice
#pragma unroll
            for (int kk = 0; kk < kTileM / 16; ++kk)
              mma_ts_by(leader, tmem + Cfg::kColDV, tmem + Cfg::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                     do_mn + kk * (2048 >> 4), kIdDV, (it > 0 || kk > 0));
          }
          mma_commit_by(leader, smem_addr(&bars->do_empty));  // dO_i fully read: the next one may load
          // S^T of the next query tile into the same TMEM columns (the MMAs run
          // in issue order, so dV has read P^T before they are overwritten)
          if (kQS == 2 && it + 1 < n_it && !(ok = wait_issue_s(it + 1))) break;
          // dK += dS^T Q (dS^T: the shared-memory dS buffer read K-major);
          // dQ = dS K (the same buffer read MN-major)
          if (!(ok = mbar_wait_warp(smem_addr(&bars->ds_ready), it & 1, lim))) break;
          tc_fence_after();
          const uint64_t qmn = q_mn + stage * kStageStep;
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            mma_ss_by(leader, tmem + Cfg::kColDK, ds_km + koff(kk), qmn + kk * (2048 >> 4), kIdDK,
                   (it > 0 || kk > 0));
          if constexpr (kQS == 1) mma_commit_by(leader, smem_addr(&bars->q_empty[0]));  // Q_i fully read
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ss_by(leader, tmem + Cfg::kColDP, ds_mn + kk * (2048 >> 4), k_mn + kk * (2048 >> 4),
                      kIdDQ, kk > 0);
          mma_commit_by(leader, smem_addr(&bars->dq_full));  // covers every earlier MMA, dV included
          if constexpr (kQS == 2) mma_commit_by(leader, smem_addr(&bars->q_empty[stage]));
          if (kQS == 1 && it + 1 < n_it && !(ok = wait_issue_s(it + 1))) break;
          // dP^T of the next tile reuses the dQ columns once dQ_i has been read out
          if (it + 1 < n_it) {
            if (!(ok = mbar_wait_warp(smem_addr(&bars->dq_free), it & 1, lim))) break;
            if (!(ok = mbar_wait_warp(smem_addr(&bars->do_full), (it + 1) & 1, lim))) break;
            tc_fence_after();
            issue_dp(it + 1);
          }
        }
        if (!ok && leader) record_error(p.err, kErrTimeout);
      }
    }
    __syncwarp();
  } else if (warp < 12) {
    regs_inc<128>();
    // --------------------------------------------------------- compute
    // Thread (warpgroup c, lane row r) owns key row r and query columns
    // [64c, 64c + 64) of S^T, P^T, dP^T and dS^T.
    const int c = (warp - 4) >> 2;
    const int r = (tid - 128) & 127;
    const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
    const int kv = t.j * kTileN + r;       // sequence-relative key row
    const bool kv_ok = kv < t.Lk;
    const float sc = p.scale_log2;
    const float* stat = reinterpret_cast<const float*>(smem + Cfg::kStatOff);
    uint8_t* ds_blk = smem + Cfg::kdSOff + c * 16384;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int stage = it % kQS;
      const int i = bwd_query_tile<SPT>(p, t, it % n_per_head);
      if (!(ok = mbar_wait(smem_addr(&bars->q_full[stage]), (it / kQS) & 1, lim))) break;
      if (!(ok = mbar_wait(smem_addr(&bars->s_full), it & 1, lim))) break;
      tc_fence_after();
      const float* lse2 = stat + stage * 256 + 64 * c;
      const float* dvs = stat + stage * 256 + 128 + 64 * c;
      float pr[64];
      {
        uint32_t sr[64];
        tmem_ld32(tmem + lane_base + Cfg::kColS + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld32(tmem + lane_base + Cfg::kColS + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        const bool diag = p.causal && (i == t.j);
#pragma unroll
        for (int q = 0; q < 64; q += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(lse2 + q);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pv = ex2_approx(fmaf(__uint_as_float(sr[q + e]), sc, -lv[e]));
            if (diag && (r > 64 * c + q + e)) pv = 0.f;  // key after query: masked
            pr[q + e] = kv_ok ? pv : 0.f;
          }
        }
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(pr[2 * e], pr[2 * e + 1]);
        // P^T (bf16 pairs) for query columns [64c, 64c+64) goes into the first
        // 32 of this warpgroup's own 64 S^T columns, so it never overwrites scores
        // the other warpgroup has still to read.
        tmem_st32(tmem + lane_base + Cfg::kColS + 64 * c, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_addr(&bars->p_ready));
      // dS^T = P^T o (dP^T - D)
      if (!(ok = mbar_wait(smem_addr(&bars->dp_full), it & 1, lim))) break;
      // dK_{i-1} and dQ_{i-1} read dS from shared memory; they must have finished
      if (it > 0 && !(ok = mbar_wait(smem_addr(&bars->dq_full), (it - 1) & 1, lim))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dp[32];
        tmem_ld32(tmem + lane_base + Cfg::kColDP + 64 * c + 32 * cc, dp);
        tmem_ld_wait(dp);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int q0 = 32 * cc + 4 * e;
          const float4 d4 = *reinterpret_cast<const float4*>(dvs + q0);
          w[2 * e] = pack_bf16x2(pr[q0] * (__uint_as_float(dp[4 * e]) - d4.x),
                                 pr[q0 + 1] * (__uint_as_float(dp[4 * e + 1]) - d4.y));
          w[2 * e + 1] = pack_bf16x2(pr[q0 + 2] * (__uint_as_float(dp[4 * e + 2]) - d4.z),
                                     pr[q0 + 3] * (__uint_as_float(dp[4 * e + 3]) - d4.w));
        }
        // dS (row r = key, 64 query columns of block c) in 128-byte-swizzled form:
        // read MN-major it is the A operand of dQ = dS K, read K-major the A
        // operand of dK = dS^T Q.
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
          *reinterpret_cast<uint4*>(ds_blk + sw128_offset(r, cc * 4 + ch)) =
              make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
      }
      fence_async_shared();
      tc_fence_before();
      mbar_arrive(smem_addr(&bars->ds_ready));
    }
    if (!ok) record_error(p.err, kErrTimeout);
    // --------------------------------------------------------- dK / dV epilogue
    // warpgroup c writes the pass's dK columns [C0 + c NC/2, C0 + (c+1) NC/2) and,
    // in the pass with dV, dV columns [c DV/2, (c+1) DV/2) of this key row
    bool have = ok && n_it > 0;
    if (have) {
      // the last dq_full commit covers every MMA, the last dV included
      have = mbar_wait(smem_addr(&bars->dq_full), (n_it - 1) & 1, lim);
      if (!have) record_error(p.err, kErrTimeout);
      tc_fence_after();
    }
    {
      // every lane takes part in the (warp-collective) TMEM loads. A whole key
      // tile leaves through shared memory (the Q stages hold dK, the dS buffer
      // dV: every MMA is done) and TMA stores of 128 x 64 boxes; the last tile
      // of a packed sequence row by row, only rows inside the sequence (a
      // 128-row box would also write the next sequence's rows)
      const bool tma_epi = !(p.cu_seqlens != nullptr && (t.j + 1) * kTileN > t.Lk);
      const size_t grow = static_cast<size_t>(t.row_base) + kv;
      const size_t krow = p.cu_seqlens ? grow * p.H_kv + t.h_kv
                                       : (static_cast<size_t>(t.b) * p.N_k + kv) * p.H_kv + t.h_kv;
      uint4* dk_row = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dk) + krow * DQK + C0);
      uint4* dv_row = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dv) + krow * DV);
      uint8_t* const stage_dk = smem + Cfg::kQOff;
      uint8_t* const stage_dv = smem + Cfg::kdSOff;
#pragma unroll
      for (int which = kDoDV ? 0 : 1; which < 2; ++which) {
        const uint32_t col = which ? Cfg::kColDK : Cfg::kColDV;
        const float mul = which ? p.scale : 1.0f;
        uint4* dst = which ? dk_row : dv_row;
        uint8_t* stg = which ? stage_dk : stage_dv;
        constexpr int kHalfMax = (NC > DV ? NC : DV) / 2;
        const int half = which ? NC / 2 : DV / 2;
        uint32_t v[kHalfMax];
        if (have) {
#pragma unroll
          for (int cc = 0; cc < kHalfMax / 32; ++cc)
            if (cc < half / 32)
              tmem_ld32(tmem + lane_base + col + c * half + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(v + cc * 32));
#pragma unroll
          for (int cc = 0; cc < kHalfMax / 32; ++cc)
            if (cc < half / 32) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + cc * 32));
        } else {
#pragma unroll
          for (int e = 0; e < kHalfMax; ++e) v[e] = 0u;
        }
#pragma unroll
        for (int e = 0; e < kHalfMax / 8; ++e) {
          if (e >= half / 8) continue;
          const uint4 w = make_uint4(
              pack_bf16x2(__uint_as_float(v[8 * e + 0]) * mul, __uint_as_float(v[8 * e + 1]) * mul),
              pack_bf16x2(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul),
              pack_bf16x2(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul),
              pack_bf16x2(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul));
          const int c8 = c * half + 8 * e;  // first column of these eight in the pass's columns
          if (tma_epi)
            *reinterpret_cast<uint4*>(stg + (c8 >> 6) * 16384 + sw128_offset(r, (c8 & 63) >> 3)) = w;
          else if (kv_ok)
            dst[c8 / 8] = w;
        }
      }
      if (tma_epi) {
        fence_async_shared();
        named_bar_sync(2, 256);  // both compute warpgroups' rows are in place
        if (c == 0 && r == 0) {
          const int row = t.row_base + t.j * kTileN;
#pragma unroll
          for (int b = 0; b < NC / 64; ++b)
            tma_store_4d(&tm_dk, smem_addr(stage_dk + b * 16384), C0 + b * 64, t.h_kv, row,
                         t.batch_coord);
          if constexpr (kDoDV) {
#pragma unroll
            for (int b = 0; b < DV / 64; ++b)
              tma_store_4d(&tm_dv, smem_addr(stage_dv + b * 16384), b * 64, t.h_kv, row,
                           t.batch_coord);
          }
          bulk_commit_group();
          bulk_wait_group<0>();  // read and written before the CTA's shared memory goes
        }
      }
    }
  } else {
    regs_inc<144>();
    // --------------------------------------------------------- dQ (query row r)
    const int r = tid - 384;
    const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int h = t.h_kv * p.group + it / n_per_head;
      const int i = bwd_query_tile<SPT>(p, t, it % n_per_head);
      if (!(ok = mbar_wait(smem_addr(&bars->dq_full), it & 1, lim))) break;
      tc_fence_after();
      uint32_t v[NC];
#pragma unroll
      for (int cc = 0; cc < NC / 32; ++cc)
        tmem_ld32(tmem + lane_base + Cfg::kColDP + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(v + cc * 32));
#pragma unroll
      for (int cc = 0; cc < NC / 32; ++cc) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + cc * 32));
      tc_fence_before();
      mbar_arrive(smem_addr(&bars->dq_free));
      int* sem = nullptr;
      if (p.deterministic) {
        // wait until every key tile ahead of this one in query tile i's order
        // has added into it
        sem = p.sem + (static_cast<size_t>(t.sem_base) + i) * p.H_q + h;
        if (r == 0) {
          const long long t0 = clock64();
          const int turn = SPT ? it % n_per_head : t.j;
          while (ld_acquire(sem) != turn) {
            if (clock64() - t0 > lim) { record_error(p.err, kErrTimeout); break; }
          }
        }
        named_bar_sync(1, 128);
      }
      if (p.cu_seqlens != nullptr && (i + 1) * kTileM > t.Lq) {
        // last tile of a packed sequence: a 128-row bulk reduction would also
        // touch the next sequence's rows, so add the valid rows one by one
        const int q = i * kTileM + r;
        if (q < t.Lq) {
          float* dst = p.dq_acc + ((static_cast<size_t>(t.row_base) + q) * p.H_q + h) * DQK + C0;
#pragma unroll
          for (int e = 0; e < NC / 4; ++e)
            red_add_v4(dst + 4 * e, __uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                       __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
        }
      } else {
        // 32 fp32 columns at a time: registers -> swizzled staging buffer ->
        // one bulk tensor reduction (rows past the end of a fixed-length batch
        // entry fall outside the tensor map and are dropped)
#pragma unroll
        for (int cc = 0; cc < NC / 32; ++cc) {
          const int buf = cc & 1;
          uint8_t* stage_buf = smem + Cfg::kdQOff + buf * 16384;
          if (r == 0) bulk_wait_group_read<1>();  // this buffer's previous reduction has read it
          named_bar_sync(1, 128);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(stage_buf + sw128_offset(r, ch)) =
                make_uint4(v[cc * 32 + 4 * ch], v[cc * 32 + 4 * ch + 1], v[cc * 32 + 4 * ch + 2],
                           v[cc * 32 + 4 * ch + 3]);
          fence_async_shared();
          named_bar_sync(1, 128);
          if (r == 0) {
            tma_reduce_add_4d(&tm_dq, smem_addr(stage_buf), C0 + cc * 32, h, t.row_base + i * kTileM,
                              t.batch_coord);
            bulk_commit_group();
          }
        }
      }
      if (p.deterministic) {
        if (r == 0) {
          bulk_wait_group<0>();  // our reductions are complete in global memory
          fence_async_global();
        }
        __threadfence();
        named_bar_sync(1, 128);
        // (failure test: the first work item never releases, so later key tiles
        // of the same query tiles give up waiting after the wait limit)
        const bool skip = p.fault == kFaultSkipDqRelease && bars->work_idx == 0;
        if (r == 0 && !skip) atomicAdd(sem, 1);
      }
    }
    if (r == 0) bulk_wait_group<0>();  // staging buffers are read before the CTA exits
    if (!ok) record_error(p.err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

cudaError_t launch_attn_bwd_pair_main(const BwdParams& p, const CUtensorMap* maps, int n_pairs,
                                      int* ticket, cudaStream_t st);

template <int DQK, int DV, int C0, int NC>
static cudaError_t launch_bwd_main(const BwdParams& p, const CUtensorMap* maps, int* ticket,
                                   int n_work, int prof_id, cudaStream_t st) {
  using Cfg = BwdCfg<DQK, DV, NC>;
  auto kern = p.spt ? attn_bwd_main_kernel<DQK, DV, C0, NC, true>
                    : attn_bwd_main_kernel<DQK, DV, C0, NC, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int slot = prof_begin(prof_id, st);
  kern<<<n_work, 512, Cfg::kSmemBytes, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[7],
                                              maps[8], p, ticket);
  e = cudaGetLastError();
  prof_end(slot, st);
  return e;
}

// n_sem: ordering semaphores of one pass (deterministic mode); each pass has
// its own set, followed by its work-ticket counter.
template <int DQK, int DV>
static cudaError_t launch_bwd_impl(const BwdParams& p, const CUtensorMap* maps, cudaStream_t st,
                                   long long rows_q, int n_sem, int n_work) {
  constexpr int kPasses = DQK > 128 ? 2 : 1;
  const long long n_rowheads = rows_q * p.H_q;
  const long long n_acc4 = n_rowheads * DQK / 4;
  const int threads = 256;
  long long want = (n_acc4 + threads - 1) / threads;
  int blocks = static_cast<int>(want < 152 * 16 ? (want > 0 ? want : 1) : 152 * 16);
  int slot = prof_begin(kKBwdPre, st);
  attn_bwd_pre_kernel<DV><<<blocks, threads, 0, st>>>(p, n_rowheads, n_acc4,
                                                      kPasses * (n_sem + 1) - 1);
  cudaError_t e = cudaGetLastError();
  prof_end(slot, st);
  if (e != cudaSuccess) return e;
  if (n_work > 0 && DQK == 128 && DV == 128 && p.pairs) {
    // CTA pairs: n_work pairs of 256 keys
    int* ticket = p.deterministic ? p.sem + n_sem : nullptr;
    e = launch_attn_bwd_pair_main(p, maps, n_work, ticket, st);
    if (e != cudaSuccess) return e;
  } else if (n_work > 0) {
    int* ticket = p.deterministic ? p.sem + n_sem : nullptr;
    e = launch_bwd_main<DQK, DV, 0, (DQK < 128 ? DQK : 128)>(p, maps, ticket, n_work, kKBwdMain, st);
    if (e != cudaSuccess) return e;
    if constexpr (kPasses == 2) {
      // query/key head columns 128 .. DQK - 1: S and dP recomputed, dK and dQ
      // for those columns, no dV
      BwdParams p1 = p;
      if (p.deterministic) p1.sem = p.sem + (n_sem + 1);
      e = launch_bwd_main<DQK, DV, 128, DQK - 128>(p1, maps, p.deterministic ? p1.sem + n_sem : nullptr,
                                                  n_work, kKBwdMain2, st);
      if (e != cudaSuccess) return e;
    }
  }
  const long long n_vec8 = n_rowheads * DQK / 8;
  want = (n_vec8 + threads - 1) / threads;
  blocks = static_cast<int>(want < 152 * 16 ? (want > 0 ? want : 1) : 152 * 16);
  slot = prof_begin(kKBwdPost, st);
  attn_bwd_post_kernel<<<blocks, threads, 0, st>>>(p, n_vec8);
  e = cudaGetLastError();
  prof_end(slot, st);
  return e;
}

// Supported (d_qk, d_v): (64, 64), (128, 128), (192, 128); the caller checks.
cudaError_t launch_attn_bwd(const BwdParams& p, const CUtensorMap* maps, cudaStream_t stream,
                            long long rows_q, int n_sem, int n_work) {
  if (p.d == 64) return launch_bwd_impl<64, 64>(p, maps, stream, rows_q, n_sem, n_work);
  if (p.d == 192) return launch_bwd_impl<192, 128>(p, maps, stream, rows_q, n_sem, n_work);
  return launch_bwd_impl<128, 128>(p, maps, stream, rows_q, n_sem, n_work);
}

}  // namespace attn

// Forward pass on CTA pairs (d = 128): the 2-CTA tensor-core mode of the
// FlashAttention-4 summary (section 2.2, and the M = 256 column of Table 1),
// kept as a selectable variant next to the one-CTA kernel in attn_fwd.cu.
//
// A cluster of two CTAs owns a block of 512 query rows of one (batch, query
// head). Each CTA holds two 128-row query tiles; tile s of the even CTA and tile
// s of the odd CTA form super tile s (256 rows). One thread of the even CTA
// issues cta_group::2 MMAs over the pair:
//   S_s  = Q_s K_j^T  with the 128 keys of K_j split 64 / 64 between the CTAs
//                     (each CTA supplies its own 128 query rows as A and 64 keys
//                     as its half of B);
//   O_s += P_s V_j    with the 128 head-dimension columns of V_j split 64 / 64
//                     (P comes from each CTA's own TMEM).
// Each instruction does twice the work of a one-CTA instruction, and each CTA
// loads into its shared memory only half of every K and V tile. Softmax, the
// lazy rescale and the epilogue run per CTA exactly as in the one-CTA kernel.
//
// Synchronisation: the TMA loads of both CTAs and the softmax arrivals of both
// CTAs are counted on the even CTA's barriers (its MMA thread is the only
// waiter); the pair commits arrive on the barrier at the same offset in both
// CTAs, so each CTA's producer and softmax warps wait on local barriers.
//
// Warp roles (384 threads per CTA): warp 0 TMA producer, warp 1 TMEM owner and
// (even CTA) MMA issuer, warps 4-7 softmax of tile 0, warps 8-11 of tile 1.
// TMEM (512 columns per CTA): O_0 [0, 128), O_1 [128, 256), S_0/P_0 [256, 384),
// S_1/P_1 [384, 512).
//
// Work: one pair per 512-row block; grid = (2 x blocks, H_q, B) for fixed
// length and (2 x upper bound on blocks, H_q, 1) for packed sequences. Causal
// masks run a batch entry's blocks longest first.
#include <cstdint>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "fwd_softmax.cuh"

namespace attn {

struct PairFwdCfg {
  static constexpr int D = 128;
  static constexpr int kQTileBytes = kTileM * D * 2;   // 32 KB
  static constexpr int kHalfBytes = 16384;             // 64 keys x 128 cols, or 128 keys x 64 cols
  static constexpr int kStages = 8;                    // ring of K / V halves
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kQTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kHalfBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kColO0 = 0, kColO1 = D;
  static constexpr uint32_t kColS0 = 2 * D, kColS1 = 2 * D + 128;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kBlockRows = 4 * kTileM;         // query rows per pair
};
static_assert(PairFwdCfg::kSmemBytes <= 232448, "shared memory");

struct PairFwdBars {
  uint64_t q_full;        // even CTA: Q tiles of both CTAs
  uint64_t s_full[2];     // both CTAs (pair commit)
  uint64_t p_full[2];     // even CTA: softmax threads of both CTAs
  uint64_t pv_done[2];    // both CTAs (pair commit)
  uint64_t kv_full[8];    // even CTA: K / V halves of both CTAs
  uint64_t kv_empty[8];   // both CTAs (pair commit)
  uint32_t tmem_base;
};

struct PairFwdTile {
  int b, h, h_kv;
  int q0;          // first query row of the 512-row block (sequence relative)
  int my0[2];      // first row of this CTA's tile s
  int row_base, batch_coord, Lq, Lk;
  int n[2];        // key tiles of super tile s (union over both CTAs' rows)
  int valid[2];    // this CTA's tile s has rows inside the sequence
};

// Both CTAs of a pair decode the same block (blockIdx.x >> 1).
__device__ __forceinline__ bool decode_pair_fwd_tile(const FwdParams& p, uint32_t rank,
                                                     PairFwdTile& t) {
  constexpr int R = PairFwdCfg::kBlockRows;
  t.h = blockIdx.y;
  t.h_kv = t.h / p.group;
  const int pidx = static_cast<int>(blockIdx.x >> 1);
  int m;
  if (p.cu_seqlens == nullptr) {
    const int nb = (p.N_q + R - 1) / R;
    if (pidx >= nb) return false;
    t.b = blockIdx.z;
    m = p.causal ? (nb - 1 - pidx) : pidx;
    t.row_base = 0;
    t.batch_coord = t.b;
    t.Lq = p.N_q;
    t.Lk = p.N_k;
  } else {
    // sequences in order, each clamped after the one before it (seq_span)
    int idx = pidx, s = 0, L = 0, nb = 0;
    SeqSpan sp{0, 0};
    for (; s < p.B; ++s) {
      sp = seq_span(p.cu_seqlens, s, p.N_q, sp.start + sp.len);
      L = sp.len;
      nb = (L + R - 1) / R;
      if (idx < nb) break;
      idx -= nb;
    }
    if (s >= p.B) return false;
    m = p.causal ? (nb - 1 - idx) : idx;
    t.b = s;
    t.row_base = sp.start;
    t.batch_coord = 0;
    t.Lq = L;
    t.Lk = L;
  }
  t.q0 = m * R;
  for (int s = 0; s < 2; ++s) {
    const int r0 = t.q0 + s * 2 * kTileM;  // first row of super tile s
    int kv_end = t.Lk;
    if (p.causal) kv_end = min(kv_end, r0 + 2 * kTileM);
    t.n[s] = (r0 < t.Lq) ? (kv_end + kTileN - 1) / kTileN : 0;
    t.my0[s] = r0 + static_cast<int>(rank) * kTileM;
    t.valid[s] = t.my0[s] < t.Lq;
  }
  return true;
}

// Epilogue of one query row: O / l and m ln 2 + ln l from the O columns in
// TMEM, or O = 0 and LSE = -inf when the row saw no key (have_o false). Every
// lane of the warp calls it: tcgen05.ld is a warp-collective instruction, so
// have_o must be the same in all lanes, and only the global stores depend on
// the lane's own row_ok.
__device__ __forceinline__ void pair_fwd_store_row(const FwdParams& p, const PairFwdTile& t,
                                                   int qrow, bool row_ok, uint32_t o_tmem,
                                                   bool have_o, float m_used, float l) {
  constexpr int D = PairFwdCfg::D;
  const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
  const size_t grow = static_cast<size_t>(t.row_base) + qrow;  // packed row
  const size_t o_off = p.cu_seqlens
                           ? (grow * p.H_q + t.h) * D
                           : ((static_cast<size_t>(t.b) * p.N_q + qrow) * p.H_q + t.h) * D;
  uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + o_off);
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t ov[32];
    if (have_o) {
      tmem_ld32(o_tmem + cc * 32, ov);
      tmem_ld_wait(ov);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) ov[e] = 0u;
    }
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      w[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
    if (row_ok) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        orow[cc * 4 + e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    }
  }
  if (row_ok) {
    const float lse = (have_o && l > 0.0f) ? (m_used * kLn2 + __logf(l)) : -INFINITY;
    const size_t l_off = p.cu_seqlens ? static_cast<size_t>(t.h) * p.N_q + grow
                                      : (static_cast<size_t>(t.b) * p.H_q + t.h) * p.N_q + qrow;
    p.lse[l_off] = lse;
  }
}

template <int EMU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_khalf,
                     const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Cfg = PairFwdCfg;
  constexpr int D = Cfg::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  PairFwdBars* bars = reinterpret_cast<PairFwdBars*>(smem + Cfg::kBarOff);
  const uint32_t rank = cluster_ctarank();

  // the first CTA reports an inconsistent packed-sequence offset array (every
  // CTA clamps what it decodes, so it stays inside the tensors either way)
  if (p.cu_seqlens != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
    check_cu_seqlens(p.cu_seqlens, p.B, p.N_q, p.err, threadIdx.x, blockDim.x);
  PairFwdTile t;
  if (!decode_pair_fwd_tile(p, rank, t)) return;  // both CTAs of the pair leave together

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    mbar_init(smem_addr(&bars->q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&bars->s_full[i]), 1);
      mbar_init(smem_addr(&bars->p_full[i]), 2 * kTileM);  // softmax threads of both CTAs
      mbar_init(smem_addr(&bars->pv_done[i]), 1);
    }
    for (int i = 0; i < Cfg::kStages; ++i) {
      mbar_init(smem_addr(&bars->kv_full[i]), 1);
      mbar_init(smem_addr(&bars->kv_empty[i]), 1);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(&bars->tmem_base), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // the barriers of both CTAs exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int n_kv = max(t.n[0], t.n[1]);
  const long long lim = p.wait_limit;

  if (warp < 4) {
    regs_dec<88>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0 && n_kv > 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_khalf);
        tma_prefetch_desc(&tm_v);
        const uint32_t qbar = cluster_map(smem_addr(&bars->q_full), 0);
        const int nq = (t.n[0] > 0) + (t.n[1] > 0);
        if (rank == 0) mbar_arrive_expect_tx(smem_addr(&bars->q_full), 2 * nq * Cfg::kQTileBytes);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (t.n[s] == 0) continue;
          const uint32_t dst = smem_addr(smem + Cfg::kQOff + s * Cfg::kQTileBytes);
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_4d_pair(dst + hf * 16384, &tm_q, qbar, hf * 64, t.h, t.row_base + t.my0[s],
                             t.batch_coord);
        }
        // ring order K_0 V_0 K_1 V_1 ...: stage it % kStages holds this CTA's half
        for (int it = 0; it < 2 * n_kv; ++it) {
          const int j = it >> 1;
          const int stage = it % Cfg::kStages;
          const int round = it / Cfg::kStages;
          if (!mbar_wait(smem_addr(&bars->kv_empty[stage]), (round & 1) ^ 1, lim)) {
            record_error(p.err, kErrTimeout);
            break;
          }
          const uint32_t fbar = smem_addr(&bars->kv_full[stage]);
          if (rank == 0) mbar_arrive_expect_tx(fbar, 2 * Cfg::kHalfBytes);
          const uint32_t fbar0 = cluster_map(fbar, 0);
          const uint32_t dst = smem_addr(smem + Cfg::kKVOff + stage * Cfg::kHalfBytes);
          if ((it & 1) == 0) {
            // K_j rows [64 rank, 64 rank + 64): two 64-column blocks of 8 KB
            for (int hf = 0; hf < D / 64; ++hf)
              tma_load_4d_pair(dst + hf * 8192, &tm_khalf, fbar0, hf * 64, t.h_kv,
                               t.row_base + j * kTileN + 64 * static_cast<int>(rank), t.batch_coord);
          } else {
            // V_j, all 128 keys, head-dimension columns [64 rank, 64 rank + 64)
            tma_load_4d_pair(dst, &tm_v, fbar0, 64 * static_cast<int>(rank), t.h_kv,
                             t.row_base + j * kTileN, t.batch_coord);
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      if (rank == 0 && n_kv > 0) {
        // the whole warp runs the issue loop; one elected lane issues each
        // MMA and commit
        const bool issuer = elect_one_sync();
        constexpr uint32_t kIdS = make_idesc_bf16(256, 128, 0, 0);
        constexpr uint32_t kIdPV = make_idesc_bf16(256, D, 0, 1);
        const uint32_t q_base = smem_addr(smem + Cfg::kQOff);
        const uint32_t kv_base = smem_addr(smem + Cfg::kKVOff);
        bool ok = mbar_wait_cluster_warp(smem_addr(&bars->q_full), 0, lim);
        const uint64_t q_desc = make_sdesc_sw128(q_base, 16, 1024);      // K-major, 128 rows
        const uint64_t k_desc = make_sdesc_sw128(kv_base, 16, 1024);     // K-major, 64 rows
        const uint64_t v_desc = make_sdesc_sw128(kv_base, 16384, 1024);  // MN-major, 64 columns
        auto stage_of = [](int it) { return it % Cfg::kStages; };
        auto phase_of = [](int it) { return (it / Cfg::kStages) & 1; };
        auto issue_s = [&](int s, int stage) {
          const uint64_t qa = q_desc + ((s * Cfg::kQTileBytes) >> 4);
          const uint64_t kb = k_desc + ((stage * Cfg::kHalfBytes) >> 4);
          const uint32_t d_tmem = tmem + Cfg::kColS0 + s * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // Q: 16 KB per 64-column block of 128 rows; K half: 8 KB per block of 64 rows
            mma_ss_pair_by(issuer, d_tmem, qa + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                        kb + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), kIdS, kk > 0);
          }
          mma_commit_pair_by(issuer, smem_addr(&bars->s_full[s]));
        };
        auto issue_pv = [&](int s, int stage, int j) {
          const uint64_t vb = v_desc + ((stage * Cfg::kHalfBytes) >> 4);
          const uint32_t d_tmem = tmem + Cfg::kColO0 + s * D;
          const uint32_t a_tmem = tmem + Cfg::kColS0 + s * 128;
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ts_pair_by(issuer, d_tmem, a_tmem + kk * 8, vb + kk * (2048 >> 4), kIdPV, (j > 0 || kk > 0));
          if (j + 1 == t.n[s]) mma_commit_pair_by(issuer, smem_addr(&bars->pv_done[s]));
        };
        if (ok) ok = mbar_wait_cluster_warp(smem_addr(&bars->kv_full[stage_of(0)]), phase_of(0), lim);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int s = 0; s < 2; ++s)
            if (t.n[s] > 0) issue_s(s, stage_of(0));
          mma_commit_pair_by(issuer, smem_addr(&bars->kv_empty[stage_of(0)]));
        }
        for (int j = 0; ok && j < n_kv; ++j) {
          const int itv = 2 * j + 1, itk = 2 * j + 2;
          const bool next_k = (j + 1) < n_kv;
          ok = mbar_wait_cluster_warp(smem_addr(&bars->kv_full[stage_of(itv)]), phase_of(itv), lim);
          if (ok && next_k)
            ok = mbar_wait_cluster_warp(smem_addr(&bars->kv_full[stage_of(itk)]), phase_of(itk), lim);
          if (!ok) break;
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            if (j >= t.n[s]) continue;
            if (!mbar_wait_cluster_warp(smem_addr(&bars->p_full[s]), j & 1, lim)) { ok = false; break; }
            tc_fence_after();
            issue_pv(s, stage_of(itv), j);
            if (j + 1 < t.n[s]) issue_s(s, stage_of(itk));
          }
          if (!ok) break;
          mma_commit_pair_by(issuer, smem_addr(&bars->kv_empty[stage_of(itv)]));
          if (next_k) mma_commit_pair_by(issuer, smem_addr(&bars->kv_empty[stage_of(itk)]));
        }
        if (!ok && issuer) record_error(p.err, kErrTimeout);
      }
    }
    __syncwarp();
  } else {
    regs_inc<208>();
    // ---------------------------------------------------------- softmax + epilogue
    const int s = (warp - 4) >> 2;          // super tile of this warpgroup
    const int r = tid - 128 * (1 + s);      // row within this CTA's tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((r & ~31)) << 16;
    const uint32_t col_s = s ? Cfg::kColS1 : Cfg::kColS0;
    const uint32_t col_o = s ? Cfg::kColO1 : Cfg::kColO0;
    const int my0 = s ? t.my0[1] : t.my0[0];
    const int qrow = my0 + r;                // sequence-relative query row
    const int my_n = s ? t.n[1] : t.n[0];
    const int my_valid = s ? t.valid[1] : t.valid[0];
    const uint32_t pbar = cluster_map(smem_addr(&bars->p_full[s]), 0);
    const float c = p.scale_log2;
    float m_used = -INFINITY;
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < my_n; ++j) {
      if (!mbar_wait(smem_addr(&bars->s_full[s]), j & 1, lim)) { ok = false; break; }
      tc_fence_after();
      float sv[128];
      {
        uint32_t* sr = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          tmem_ld32(tmem + lane_base + col_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + cc * 32));
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sr + cc * 32));
      }
      const int kv0 = j * kTileN;
      const bool need_mask = (kv0 + kTileN > t.Lk) || (p.causal && kv0 + kTileN - 1 > my0);
      uint32_t pk[64];
      bool rescale_warp;
      float factor;
      if (c > 0.0f)
        softmax_row_tile<EMU, true>(sv, c, m_used, l, kv0, qrow, t.Lk, need_mask, p.causal, pk,
                                    rescale_warp, factor);
      else
        softmax_row_tile<0, false>(sv, c, m_used, l, kv0, qrow, t.Lk, need_mask, p.causal, pk,
                                   rescale_warp, factor);
      if (rescale_warp && j > 0 && __any_sync(0xffffffffu, factor != 1.0f)) {
        // O_{j-1} is complete: the commit that signalled S_j followed its PV
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + col_o + cc * 32, ov);
          tmem_ld_wait(ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
          tmem_st32(tmem + lane_base + col_o + cc * 32, ov);
        }
      }
      tmem_st32(tmem + lane_base + col_s, *reinterpret_cast<uint32_t(*)[32]>(pk));
      tmem_st32(tmem + lane_base + col_s + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_cluster(pbar);  // the even CTA's MMA thread waits for both CTAs
    }
    if (!ok) record_error(p.err, kErrTimeout);
    // ---------------------------------------------------------- epilogue
    bool have_o = ok && my_n > 0;
    if (have_o) {
      have_o = mbar_wait(smem_addr(&bars->pv_done[s]), 0, lim);
      if (!have_o) record_error(p.err, kErrTimeout);
      tc_fence_after();
    }
    // my_n and my_valid are the same for the whole warpgroup; a wait that gave
    // up in one lane drops the O loads of its warp
    have_o = __all_sync(0xffffffffu, have_o);
    if (my_valid) pair_fwd_store_row(p, t, qrow, qrow < t.Lq, tmem + lane_base + col_o, have_o, m_used, l);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the pair's MMAs read both CTAs' shared memory and TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, Cfg::kTmemCols);
  }
}

#ifndef ATTN_FWD_EMU
#define ATTN_FWD_EMU 0
#endif

// grid.x = 2 x (512-row blocks); tk_half maps 64-row K boxes.
cudaError_t launch_attn_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tk_half,
                                 const CUtensorMap& tv, const FwdParams& p, dim3 grid,
                                 cudaStream_t stream) {
  auto kern = attn_fwd_pair_kernel<ATTN_FWD_EMU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PairFwdCfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int slot = prof_begin(kKFwdPair, stream);
  kern<<<grid, 384, PairFwdCfg::kSmemBytes, stream>>>(tq, tk_half, tv, p);
  e = cudaGetLastError();
  prof_end(slot, stream);
  return e;
}

}  // namespace attn

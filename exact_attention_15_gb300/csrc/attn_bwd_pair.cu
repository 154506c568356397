// Backward main kernel on CTA pairs (d = 128): the 2-CTA backward of the
// FlashAttention-4 summary, section 3.2.3.
//
// A cluster of two CTAs owns 256 consecutive keys of one (batch, KV head):
// CTA c ("rank") holds keys [256 J + 128 c, +128) in shared memory and its dK /
// dV rows in TMEM. Both walk the same query tiles. S^T, dP^T, dV and dK run as
// M = 256 tcgen05 MMAs over the pair (cta_group::2): each CTA supplies the A
// rows of its own keys and half of operand B (Q_i or dO_i), so each CTA reads
// only half of every B tile from shared memory, which is what bounds the
// one-CTA backward. dQ = dS K reduces over the keys, which the pair splits; so
// the CTAs swap halves of dS through distributed shared memory and run dQ as an
// M = 128 pair MMA over all 256 keys: CTA c computes the dQ rows of query half
// c, and each CTA adds only 64 rows of every dQ tile to the accumulator.
//
// Operand layout. A pair MMA combines CTA 0's A rows with CTA 1's half of B
// (and the reverse), so the reduction dimension is laid out alike in both CTAs
// and each CTA keeps, at the same shared-memory offsets, the part of every B
// operand it supplies: the 64 rows of its own query half of Q_i and dO_i (B of
// S^T and dP^T, reduced over d), the 64-column block of its own half of the head
// dimension of Q_i and dO_i (B of dK and dV, reduced over the queries), and that
// column block of K for both CTAs' keys together with the dS^T rows of both
// CTAs' keys for its own query half (B and A of dQ, reduced over 256 keys).
//
// Warp roles (512 threads per CTA):
//   warp 0      producer: K, V (own keys) and the dQ key blocks, then per query
//               tile the query-half and d-block parts of Q_i and dO_i by TMA
//               (their completions counted on CTA 0's barriers) and LSE_i, D_i.
//   warp 1      CTA 0 only: issues every pair MMA.
//   warps 4-11  compute, two warpgroups: thread r of warpgroup w owns key row r
//               and query half w: P^T, dS^T, and at the end half of the dK / dV
//               row.
//   warps 12-15 dQ: TMEM -> registers -> shared memory -> bulk tensor
//               reductions of this CTA's 64 dQ rows.
//
// TMEM (512 columns per CTA): dV [0, 128), dK [128, 256), S^T / P^T [256, 384),
// dP^T / dS^T [384, 512), dQ (64 rows as 128 lanes x 64 columns) [384, 448).
#include <cstdint>
#include <climits>
#include <cuda_runtime.h>

#include "attn_common.cuh"

namespace attn {

struct PairCfg {
  static constexpr int D = 128;
  static constexpr int kTileBytes = kTileM * D * 2;       // 32 KB
  static constexpr int kBlk = 16384;                      // [128 rows x 64 cols] bf16
  static constexpr int kHalfBlk = 8192;                   // [64 rows x 64 cols] bf16
  static constexpr int kKOff = 0;                         // own keys, both d-blocks
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQrOff = kVOff + kTileBytes;       // Q_i own query half, 2 stages x 16 KB
  static constexpr int kQcOff = kQrOff + 2 * kBlk;        // Q_i own d-block, all rows
  static constexpr int kdOrOff = kQcOff + kBlk;           // dO_i own query half
  static constexpr int kdOcOff = kdOrOff + kBlk;          // dO_i own d-block
  static constexpr int kBKOff = kdOcOff + kBlk;           // K own d-block: CTA 0's keys, CTA 1's keys
  static constexpr int kRKOff = kBKOff + 2 * kBlk;        // dS^T own query half: CTA 0's keys, CTA 1's
  static constexpr int kdQOff = kRKOff + 2 * kBlk;        // 2 x (64 rows x 32 fp32) staging
  static constexpr int kStatOff = kdQOff + 2 * 8192;      // 2 stages x (lse2[128], D[128])
  static constexpr int kBarOff = kStatOff + 2 * 2 * 128 * 4;
  static constexpr int kSmemBytes = kBarOff + 256;
  static constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384;
  static constexpr uint32_t kTmemCols = 512;
};
static_assert(PairCfg::kSmemBytes <= 232448, "shared memory");

struct PairBars {
  // full barriers live in CTA 0 and count both CTAs' copies; empty barriers are
  // per CTA and signalled by the pair MMA commits
  uint64_t kv_full;                  // K, V, dQ key blocks
  uint64_t q_full[2];                // Q_i query half, per stage
  uint64_t qc_full, do_r_full, do_c_full;
  uint64_t q_empty[2], qc_empty, do_r_empty, do_c_empty;
  uint64_t st_full[2];               // local: LSE_i and D_i of a stage
  uint64_t s_full, dp_full, dq_full; // local (pair commit)
  uint64_t p_ready, ds_ready, dq_free;  // CTA 0: warps of both CTAs
  uint64_t fin;                      // local (pair commit): every MMA of the pair is done
  uint32_t tmem_base;
  int work_idx;
};

struct PairTile {
  int b, h_kv, J;
  int row_base, batch_coord, Lq, Lk;
  int k_own, k_other;   // first key (sequence relative) of this CTA / of the other CTA
  int i_start, n_qt;    // query tiles [i_start, n_qt) of each query head
  int sem_base;
};

__device__ __forceinline__ bool decode_pair_tile(const BwdParams& p, int idx, uint32_t rank,
                                                 PairTile& t) {
  if (p.cu_seqlens == nullptr) {
    const int nJ = (p.N_k + 2 * kTileN - 1) / (2 * kTileN);
    if (nJ == 0) return false;
    t.J = idx % nJ;
    const int rest = idx / nJ;
    t.h_kv = rest % p.H_kv;
    t.b = rest / p.H_kv;
    if (t.b >= p.B) return false;
    t.row_base = 0;
    t.batch_coord = t.b;
    t.Lq = p.N_q;
    t.Lk = p.N_k;
    t.sem_base = t.b * ((p.N_q + kTileM - 1) / kTileM);
  } else {
    // sequences in order, each clamped after the one before it (seq_span), so
    // their query-tile slots stay within the semaphore array
    int s = 0, qslots = 0;
    SeqSpan sp{0, 0};
    for (; s < p.B; ++s) {
      sp = seq_span(p.cu_seqlens, s, p.N_q, sp.start + sp.len);
      const int nJ = (sp.len + 2 * kTileN - 1) / (2 * kTileN);
      if (idx < nJ * p.H_kv) break;
      idx -= nJ * p.H_kv;
      qslots += (sp.len + kTileM - 1) / kTileM;
    }
    if (s >= p.B) return false;
    const int L = sp.len;
    const int nJ = (L + 2 * kTileN - 1) / (2 * kTileN);
    t.J = idx % nJ;
    t.h_kv = idx / nJ;
    t.b = s;
    t.row_base = sp.start;
    t.batch_coord = 0;
    t.Lq = L;
    t.Lk = L;
    t.sem_base = qslots;
  }
  t.k_own = 2 * kTileN * t.J + kTileN * static_cast<int>(rank);
  t.k_other = 2 * kTileN * t.J + kTileN * static_cast<int>(1 - rank);
  t.n_qt = (t.Lq + kTileM - 1) / kTileM;
  t.i_start = p.causal ? 2 * t.J : 0;  // the first query tile that sees key 256 J
  if (t.i_start > t.n_qt) t.i_start = t.n_qt;
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(512, 1)
attn_bwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_q64,
                     const __grid_constant__ CUtensorMap tm_do64, const BwdParams p, int* ticket) {
  // tm_q, tm_k, tm_v, tm_do: 128-row boxes; tm_q64, tm_do64: 64-row boxes;
  // tm_dq: fp32 dQ accumulator, 64-row x 32-column boxes
  using Cfg = PairCfg;
  constexpr int D = Cfg::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  PairBars* bars = reinterpret_cast<PairBars*>(smem + Cfg::kBarOff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();

  if ((smem_addr(smem) & 1023u) != 0) {  // same in both CTAs: both leave here
    if (tid == 0) record_error(p.err, kErrTimeout);
    return;
  }
  // Work item: CTA 0 takes a ticket in deterministic mode (so every tile a pair
  // waits on belongs to a pair that started earlier), else the cluster index;
  // CTA 1 copies it before either CTA may leave.
  if (rank == 0 && tid == 0)
    bars->work_idx = (ticket != nullptr) ? atomicAdd(ticket, 1) : static_cast<int>(blockIdx.x >> 1);
  cluster_sync_all();
  if (rank == 1 && tid == 0) bars->work_idx = ld_cluster_s32(cluster_map(smem_addr(&bars->work_idx), 0));
  cluster_sync_all();
  PairTile t;
  if (!decode_pair_tile(p, bars->work_idx, rank, t)) return;  // both CTAs alike
  const int n_per_head = t.n_qt - t.i_start;
  const int n_it = n_per_head * p.group;
  const long long lim = p.wait_limit;

  if (tid == 0) {
    mbar_init(smem_addr(&bars->kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&bars->q_full[s]), 1);
      mbar_init(smem_addr(&bars->q_empty[s]), 1);
      mbar_init(smem_addr(&bars->st_full[s]), 32);
    }
    mbar_init(smem_addr(&bars->qc_full), 1);
    mbar_init(smem_addr(&bars->do_r_full), 1);
    mbar_init(smem_addr(&bars->do_c_full), 1);
    mbar_init(smem_addr(&bars->qc_empty), 1);
    mbar_init(smem_addr(&bars->do_r_empty), 1);
    mbar_init(smem_addr(&bars->do_c_empty), 1);
    mbar_init(smem_addr(&bars->s_full), 1);
    mbar_init(smem_addr(&bars->dp_full), 1);
    mbar_init(smem_addr(&bars->dq_full), 1);
    mbar_init(smem_addr(&bars->p_ready), 16);   // 8 compute warps x 2 CTAs
    mbar_init(smem_addr(&bars->ds_ready), 16);
    mbar_init(smem_addr(&bars->dq_free), 8);    // 4 dQ warps x 2 CTAs
    mbar_init(smem_addr(&bars->fin), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(&bars->tmem_base), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers and TMEM of both CTAs exist before anyone uses them
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  auto leader = [](uint32_t local) { return cluster_map(local, 0); };
  // arrival on a barrier of CTA 0: a plain (CTA-scope) arrive there, a
  // cluster-scope release from CTA 1
  auto arrive_leader = [rank](uint32_t local, uint32_t cluster_addr) {
    if (rank == 0) mbar_arrive(local);
    else mbar_arrive_cluster(cluster_addr);
  };

  // Register split: 128 x 104 (warps 0-3) + 256 x 128 (compute) + 128 x 144 (dQ)
  // = 64,512 <= 512 x 128 (the launch total).
  if (warp < 4) {
    regs_dec<104>();
    if (warp == 0) {
      // ------------------------------------------------------- producer
      // Loads in the order the MMAs need them: per query tile it, the d-block
      // parts of dO_it and Q_it (dV_it, dK_it), then the query-half parts of
      // Q_{it+1} (S_{it+1}) with its LSE / D rows and of dO_{it+1} (dP_{it+1}).
      // Every load waits for its buffer's empty barrier (load k waits for
      // parity (k & 1) ^ 1, or ((k >> 1) & 1) ^ 1 for the two-stage Q half).
      if (n_it > 0) {
        float* stat = reinterpret_cast<float*>(smem + Cfg::kStatOff);
        const int r_own = 64 * static_cast<int>(rank);        // first row of own query half
        const int c_own = 64 * static_cast<int>(rank);        // first column of own d-block
        auto head_of = [&](int it) { return t.h_kv * p.group + it / n_per_head; };
        auto tile_of = [&](int it) { return t.i_start + it % n_per_head; };
        // arms CTA 0's full barrier for both CTAs' bytes; returns its cluster address
        auto arm = [&](uint64_t* bar, uint32_t bytes) {
          if (rank == 0) mbar_arrive_expect_tx(smem_addr(bar), 2 * bytes);
          return leader(smem_addr(bar));
        };
        auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int it) {
          // own query half of the tile, both d-blocks (64-row boxes)
          for (int blk = 0; blk < 2; ++blk)
            tma_load_4d_pair(dst + blk * Cfg::kHalfBlk, map, bar, blk * 64, head_of(it),
                             t.row_base + tile_of(it) * kTileM + r_own, t.batch_coord);
        };
        auto load_cols = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int it) {
          // own d-block of the tile, all 128 rows
          tma_load_4d_pair(dst, map, bar, c_own, head_of(it), t.row_base + tile_of(it) * kTileM,
                           t.batch_coord);
        };
        auto load_stats = [&](int it) {
          // LSE (to log2 units) and D of the 128 rows of the query tile, natural
          // order; rows past the end get LSE = +inf so that P is 0
          const int h = head_of(it), i = tile_of(it);
          float* lse2 = stat + (it & 1) * 256;
          float* dvs = lse2 + 128;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = lane + 32 * e;
            const int q = i * kTileM + r;
            float lv = INFINITY, dv = 0.f;
            if (q < t.Lq) {
              const size_t off = p.cu_seqlens
                                     ? static_cast<size_t>(h) * p.N_q + t.row_base + q
                                     : (static_cast<size_t>(t.b) * p.H_q + h) * p.N_q + q;
              lv = p.lse[off] * kLog2e;
              dv = p.dvec[off];
              if (lv == -INFINITY) lv = INFINITY;  // a row that saw no key has no gradient
            }
            lse2[r] = lv;
            dvs[r] = dv;
          }
          mbar_arrive(smem_addr(&bars->st_full[it & 1]));
        };
        bool ok = true;
        auto wait_empty = [&](uint64_t* bar, uint32_t parity) {
          if (ok && !mbar_wait(smem_addr(bar), parity, lim)) {
            record_error(p.err, kErrTimeout);
            ok = false;
          }
          return ok;
        };
        if (lane == 0) {
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_do);
          tma_prefetch_desc(&tm_q64);
          tma_prefetch_desc(&tm_do64);
          const uint32_t kvb = arm(&bars->kv_full, 2 * Cfg::kTileBytes + 2 * Cfg::kBlk);
          for (int blk = 0; blk < 2; ++blk) {
            tma_load_4d_pair(smem_addr(smem + Cfg::kKOff) + blk * Cfg::kBlk, &tm_k, kvb, blk * 64,
                             t.h_kv, t.row_base + t.k_own, t.batch_coord);
            tma_load_4d_pair(smem_addr(smem + Cfg::kVOff) + blk * Cfg::kBlk, &tm_v, kvb, blk * 64,
                             t.h_kv, t.row_base + t.k_own, t.batch_coord);
            // dQ key blocks: keys of CTA blk, own d-block
            tma_load_4d_pair(smem_addr(smem + Cfg::kBKOff) + blk * Cfg::kBlk, &tm_k, kvb, c_own,
                             t.h_kv, t.row_base + 2 * kTileN * t.J + kTileN * blk, t.batch_coord);
          }
          load_rows(smem_addr(smem + Cfg::kQrOff), &tm_q64, arm(&bars->q_full[0], Cfg::kBlk), 0);
          load_rows(smem_addr(smem + Cfg::kdOrOff), &tm_do64, arm(&bars->do_r_full, Cfg::kBlk), 0);
        }
        load_stats(0);
        for (int it = 0; it < n_it && ok; ++it) {
          if (wait_empty(&bars->do_c_empty, (it & 1) ^ 1) && lane == 0)
            load_cols(smem_addr(smem + Cfg::kdOcOff), &tm_do, arm(&bars->do_c_full, Cfg::kBlk), it);
          if (wait_empty(&bars->qc_empty, (it & 1) ^ 1) && lane == 0)
            load_cols(smem_addr(smem + Cfg::kQcOff), &tm_q, arm(&bars->qc_full, Cfg::kBlk), it);
          const int nx = it + 1;
          if (nx < n_it) {
            if (wait_empty(&bars->q_empty[nx & 1], ((nx >> 1) & 1) ^ 1)) {
              if (lane == 0)
                load_rows(smem_addr(smem + Cfg::kQrOff + (nx & 1) * Cfg::kBlk), &tm_q64,
                          arm(&bars->q_full[nx & 1], Cfg::kBlk), nx);
              load_stats(nx);
            }
            if (wait_empty(&bars->do_r_empty, (nx & 1) ^ 1) && lane == 0)
              load_rows(smem_addr(smem + Cfg::kdOrOff), &tm_do64, arm(&bars->do_r_full, Cfg::kBlk), nx);
          }
          __syncwarp();
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------- MMA issuer (CTA 0)
      // Per query tile: dV_i, S_{i+1}, dK_i, dQ_i, dP_{i+1} (after S_0, dP_0).
      if (rank == 0 && n_it > 0) {
        // the whole warp runs the issue loop; one elected lane issues each
        // MMA and commit
        const bool issuer = elect_one_sync();
        constexpr uint32_t kIdSS = make_idesc_bf16(256, 128, 0, 0);  // S^T, dP^T
        constexpr uint32_t kIdTS = make_idesc_bf16(256, D, 0, 1);    // dV, dK: B MN-major
        constexpr uint32_t kIdDQ = make_idesc_bf16(128, D, 1, 1);    // dQ: A, B MN-major
        const uint64_t k_km = make_sdesc_sw128(smem_addr(smem + Cfg::kKOff), 16, 1024);
        const uint64_t v_km = make_sdesc_sw128(smem_addr(smem + Cfg::kVOff), 16, 1024);
        const uint64_t qr_km = make_sdesc_sw128(smem_addr(smem + Cfg::kQrOff), 16, 1024);
        const uint64_t dor_km = make_sdesc_sw128(smem_addr(smem + Cfg::kdOrOff), 16, 1024);
        const uint64_t qc_mn = make_sdesc_sw128(smem_addr(smem + Cfg::kQcOff), 16384, 1024);
        const uint64_t doc_mn = make_sdesc_sw128(smem_addr(smem + Cfg::kdOcOff), 16384, 1024);
        const uint64_t bk_mn = make_sdesc_sw128(smem_addr(smem + Cfg::kBKOff), 16384, 1024);
        const uint64_t rk_mn = make_sdesc_sw128(smem_addr(smem + Cfg::kRKOff), 16384, 1024);
        // K-major steps over d: in 128-row tiles the 64-column blocks are 16 KB
        // apart, in the 64-row query halves 8 KB
        auto koff = [](int kk) { return static_cast<uint32_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
        auto koff_h = [](int kk) { return static_cast<uint32_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4); };
        auto issue_s = [&](int it) {  // S^T = K Q^T
          const uint64_t qb = qr_km + (it & 1) * (Cfg::kBlk >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_pair_by(issuer, tmem + Cfg::kColS, k_km + koff(kk), qb + koff_h(kk), kIdSS, kk > 0);
          mma_commit_pair_by(issuer, smem_addr(&bars->s_full));
        };
        auto issue_dp = [&]() {  // dP^T = V dO^T
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_pair_by(issuer, tmem + Cfg::kColDP, v_km + koff(kk), dor_km + koff_h(kk), kIdSS, kk > 0);
          mma_commit_pair_by(issuer, smem_addr(&bars->dp_full));
          mma_commit_pair_by(issuer, smem_addr(&bars->do_r_empty));
        };
        bool ok = mbar_wait_cluster_warp(smem_addr(&bars->kv_full), 0, lim);
        if (ok) ok = mbar_wait_cluster_warp(smem_addr(&bars->q_full[0]), 0, lim);
        if (ok) {
          tc_fence_after();
          issue_s(0);
        }
        if (ok) ok = mbar_wait_cluster_warp(smem_addr(&bars->do_r_full), 0, lim);
        if (ok) {
          tc_fence_after();
          issue_dp();
        }
        for (int it = 0; ok && it < n_it; ++it) {
          const int stage = it & 1;
          // dV += P^T dO: P^T of query half s sits in S^T columns [64 s, 64 s + 32)
          if (!(ok = mbar_wait_cluster_warp(smem_addr(&bars->p_ready), it & 1, lim))) break;
          if (!(ok = mbar_wait_cluster_warp(smem_addr(&bars->do_c_full), it & 1, lim))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            mma_ts_pair_by(issuer, tmem + Cfg::kColDV, tmem + Cfg::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                        doc_mn + kk * (2048 >> 4), kIdTS, (it > 0 || kk > 0));
          mma_commit_pair_by(issuer, smem_addr(&bars->do_c_empty));
          // S^T of the next query tile into the same columns (MMAs run in issue
          // order: dV has read P^T first)
          if (it + 1 < n_it) {
            if (!(ok = mbar_wait_cluster_warp(smem_addr(&bars->q_full[(it + 1) & 1]), ((it + 1) >> 1) & 1, lim)))
              break;
            tc_fence_after();
            issue_s(it + 1);
          }
          // dK += dS^T Q (dS^T in TMEM over dP^T); dQ = dS K over both CTAs' keys
          if (!(ok = mbar_wait_cluster_warp(smem_addr(&bars->ds_ready), it & 1, lim))) break;
          if (!(ok = mbar_wait_cluster_warp(smem_addr(&bars->qc_full), it & 1, lim))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            mma_ts_pair_by(issuer, tmem + Cfg::kColDK, tmem + Cfg::kColDP + (kk >> 2) * 64 + (kk & 3) * 8,
                        qc_mn + kk * (2048 >> 4), kIdTS, (it > 0 || kk > 0));
          mma_commit_pair_by(issuer, smem_addr(&bars->qc_empty));
#pragma unroll
          for (int kk = 0; kk < 2 * kTileN / 16; ++kk) {
            // key step kk: keys of CTA kk / 8, rows 16 (kk % 8) ..
            const uint32_t off = ((kk >> 3) * Cfg::kBlk + (kk & 7) * 2048) >> 4;
            mma_ss_pair_by(issuer, tmem + Cfg::kColDP, rk_mn + off, bk_mn + off, kIdDQ, kk > 0);
          }
          mma_commit_pair_by(issuer, smem_addr(&bars->dq_full));  // covers every earlier MMA, dV included
          mma_commit_pair_by(issuer, smem_addr(&bars->q_empty[stage]));
          // dP^T of the next tile reuses the dQ columns once dQ_i has been read out
          if (it + 1 < n_it) {
            if (!(ok = mbar_wait_cluster_warp(smem_addr(&bars->dq_free), it & 1, lim))) break;
            if (!(ok = mbar_wait_cluster_warp(smem_addr(&bars->do_r_full), (it + 1) & 1, lim))) break;
            tc_fence_after();
            issue_dp();
          }
        }
        // a last commit, after which no arrival of this pair's MMAs is pending
        // in either CTA
        if (ok) mma_commit_pair_by(issuer, smem_addr(&bars->fin));
        if (!ok && issuer) record_error(p.err, kErrTimeout);
      }
      if (lane == 0 && n_it > 0 && !mbar_wait(smem_addr(&bars->fin), 0, lim))
        record_error(p.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp < 12) {
    regs_inc<128>();
    // --------------------------------------------------------- compute
    // Thread (warpgroup w, lane row r) owns key row r and query half w.
    const int w = (warp - 4) >> 2;
    const int r = (tid - 128) & 127;
    const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
    const uint32_t slot = static_cast<uint32_t>(w);
    const int kv = t.k_own + r;             // sequence-relative key row
    const bool kv_ok = kv < t.Lk;
    const float sc = p.scale_log2;
    const float* stat = reinterpret_cast<const float*>(smem + Cfg::kStatOff);
    const uint32_t pbar_local = smem_addr(&bars->p_ready);
    const uint32_t dsbar_local = smem_addr(&bars->ds_ready);
    const uint32_t pbar = leader(pbar_local);
    const uint32_t dsbar = leader(dsbar_local);
    // this warpgroup's dS^T rows (this CTA's keys, query half w) go to the dQ
    // operand block of this CTA's keys in the CTA that owns query half w
    const bool ds_local = (static_cast<uint32_t>(w) == rank);
    uint8_t* ds_local_blk = smem + Cfg::kRKOff + rank * Cfg::kBlk;
    const uint32_t ds_remote_blk = cluster_map(smem_addr(ds_local_blk), 1 - rank);
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int stage = it & 1;
      const int i = t.i_start + it % n_per_head;
      if (!(ok = mbar_wait(smem_addr(&bars->st_full[stage]), (it >> 1) & 1, lim))) break;
      if (!(ok = mbar_wait(smem_addr(&bars->s_full), it & 1, lim))) break;
      tc_fence_after();
      const float* lse2 = stat + stage * 256 + 64 * w;
      const float* dvs = stat + stage * 256 + 128 + 64 * w;
      // causal: key kv sees query q only if kv <= q, i.e. column e is masked when e < thr
      const int thr = p.causal ? (kv - (i * kTileM + 64 * w)) : INT_MIN;
      float pr[64];
      {
        uint32_t sr[64];
        tmem_ld32(tmem + lane_base + Cfg::kColS + 64 * w, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld32(tmem + lane_base + Cfg::kColS + 64 * w + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sr + 32));
#pragma unroll
        for (int q = 0; q < 64; q += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(lse2 + q);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pv = ex2_approx(fmaf(__uint_as_float(sr[q + e]), sc, -lv[e]));
            if (q + e < thr) pv = 0.f;
            pr[q + e] = kv_ok ? pv : 0.f;
          }
        }
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(pr[2 * e], pr[2 * e + 1]);
        tmem_st32(tmem + lane_base + Cfg::kColS + 64 * slot, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(pbar_local, pbar);
      // dS^T = P^T o (dP^T - D)
      if (!(ok = mbar_wait(smem_addr(&bars->dp_full), it & 1, lim))) break;
      // dQ_{i-1} read both CTAs' dS blocks; it must have finished
      if (it > 0 && !(ok = mbar_wait(smem_addr(&bars->dq_full), (it - 1) & 1, lim))) break;
      tc_fence_after();
      uint32_t ws[32];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dp[32];
        tmem_ld32(tmem + lane_base + Cfg::kColDP + 64 * w + 32 * cc, dp);
        tmem_ld_wait(dp);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int q0 = 32 * cc + 4 * e;
          const float4 d4 = *reinterpret_cast<const float4*>(dvs + q0);
          ws[16 * cc + 2 * e] = pack_bf16x2(pr[q0] * (__uint_as_float(dp[4 * e]) - d4.x),
                                            pr[q0 + 1] * (__uint_as_float(dp[4 * e + 1]) - d4.y));
          ws[16 * cc + 2 * e + 1] = pack_bf16x2(pr[q0 + 2] * (__uint_as_float(dp[4 * e + 2]) - d4.z),
                                                pr[q0 + 3] * (__uint_as_float(dp[4 * e + 3]) - d4.w));
        }
      }
      // dS^T into TMEM (A operand of dK), query slot as for P^T
      tmem_st32(tmem + lane_base + Cfg::kColDP + 64 * slot, ws);
      // dS^T row r (64 queries, 128-byte-swizzled) into the dQ operand block of
      // the CTA that owns this query half
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 v = make_uint4(ws[4 * ch], ws[4 * ch + 1], ws[4 * ch + 2], ws[4 * ch + 3]);
        if (ds_local)
          *reinterpret_cast<uint4*>(ds_local_blk + sw128_offset(r, ch)) = v;
        else
          st_cluster_v4(ds_remote_blk + sw128_offset(r, ch), v);
      }
      tmem_st_wait();
      if (ds_local) fence_async_shared();
      else fence_async_shared_cluster();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(dsbar_local, dsbar);
    }
    if (!ok) record_error(p.err, kErrTimeout);
    // --------------------------------------------------------- dK / dV epilogue
    // warpgroup w writes head-dimension columns [64 w, 64 w + 64) of key row r
    bool have = ok && n_it > 0;
    if (have) {
      // the last dq_full commit covers every MMA, the last dV and dK included
      have = mbar_wait(smem_addr(&bars->dq_full), (n_it - 1) & 1, lim);
      if (!have) record_error(p.err, kErrTimeout);
      tc_fence_after();
    }
    {
      const size_t grow = static_cast<size_t>(t.row_base) + kv;
      const size_t off = p.cu_seqlens
                             ? (grow * p.H_kv + t.h_kv) * D
                             : ((static_cast<size_t>(t.b) * p.N_k + kv) * p.H_kv + t.h_kv) * D;
      uint4* dk_row = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dk) + off);
      uint4* dv_row = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dv) + off);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which ? Cfg::kColDK : Cfg::kColDV;
        const float mul = which ? p.scale : 1.0f;
        uint4* dst = which ? dk_row : dv_row;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c0 = 64 * w + cc * 32;
          uint32_t v[32];
          if (have) {
            tmem_ld32(tmem + lane_base + col + c0, v);
            tmem_ld_wait(v);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          if (kv_ok) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[c0 / 8 + e] = make_uint4(
                  pack_bf16x2(__uint_as_float(v[8 * e + 0]) * mul, __uint_as_float(v[8 * e + 1]) * mul),
                  pack_bf16x2(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul),
                  pack_bf16x2(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul),
                  pack_bf16x2(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul));
          }
        }
      }
    }
  } else {
    regs_inc<144>();
    // --------------------------------------------------------- dQ (warps 12-15)
    // An M = 128 pair MMA leaves each CTA's 64 dQ rows in 64 TMEM columns of all
    // 128 lanes: lane r holds row r % 64, columns [64 (r / 64), +64). Thread r
    // drains lane r.
    const int r = tid - 384;
    const int qr = r & 63;            // row within this CTA's query half
    const int half = r >> 6;          // which 64 of the head-dimension columns
    const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
    const uint32_t freebar_local = smem_addr(&bars->dq_free);
    const uint32_t freebar = leader(freebar_local);
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int h = t.h_kv * p.group + it / n_per_head;
      const int i = t.i_start + it % n_per_head;
      if (!(ok = mbar_wait(smem_addr(&bars->dq_full), it & 1, lim))) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(tmem + lane_base + Cfg::kColDP, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32(tmem + lane_base + Cfg::kColDP + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(freebar_local, freebar);
      const int row0 = i * kTileM + 64 * static_cast<int>(rank);  // first query row of this half
      int* sem = nullptr;
      if (p.deterministic) {
        // every earlier key pair has added both of its halves into query tile i
        sem = p.sem + (static_cast<size_t>(t.sem_base) + i) * p.H_q + h;
        if (r == 0) {
          const long long t0 = clock64();
          while (ld_acquire(sem) < 2 * t.J) {
            if (clock64() - t0 > lim) { record_error(p.err, kErrTimeout); break; }
          }
        }
        named_bar_sync(1, 128);
      }
      if (p.cu_seqlens != nullptr && row0 + 64 > t.Lq) {
        // last rows of a packed sequence: a 64-row bulk reduction would also
        // touch the next sequence's rows, so add the valid rows one by one
        const int q = row0 + qr;
        if (q < t.Lq) {
          float* dst = p.dq_acc + ((static_cast<size_t>(t.row_base) + q) * p.H_q + h) * D + 64 * half;
#pragma unroll
          for (int e = 0; e < 16; ++e)
            red_add_v4(dst + 4 * e, __uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                       __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
        }
      } else {
        // two steps of 32 columns: the half-0 threads stage columns [32 s, +32)
        // in buffer 0, the half-1 threads columns [64 + 32 s, +32) in buffer 1
        // (64 rows x 32 fp32, 128-byte swizzle); one thread of each half then
        // issues a bulk tensor reduction of its buffer (rows past the end of a
        // fixed-length batch entry fall outside the tensor map and are dropped)
        uint8_t* stage_buf = smem + Cfg::kdQOff + half * 8192;
#pragma unroll
        for (int step = 0; step < 2; ++step) {
          if (qr == 0) bulk_wait_group_read<0>();  // the previous reduction has read the buffer
          named_bar_sync(1, 128);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(stage_buf + sw128_offset(qr, ch)) =
                make_uint4(v[32 * step + 4 * ch], v[32 * step + 4 * ch + 1],
                           v[32 * step + 4 * ch + 2], v[32 * step + 4 * ch + 3]);
          fence_async_shared();
          named_bar_sync(1, 128);
          if (qr == 0) {
            tma_reduce_add_4d(&tm_dq, smem_addr(stage_buf), 64 * half + 32 * step, h,
                              t.row_base + row0, t.batch_coord);
            bulk_commit_group();
          }
        }
      }
      if (p.deterministic) {
        if (qr == 0) {
          bulk_wait_group<0>();  // our reductions are complete in global memory
          fence_async_global();
        }
        __threadfence();
        named_bar_sync(1, 128);
        // (failure test: the first work item never releases, so later key
        // pairs of the same query tiles give up waiting after the wait limit)
        const bool skip = p.fault == kFaultSkipDqRelease && bars->work_idx == 0;
        if (r == 0 && !skip) atomicAdd(sem, 1);
      }
    }
    if (qr == 0) bulk_wait_group<0>();  // staging buffers are read before the CTA exits
    if (!ok) record_error(p.err, kErrTimeout);
  }
  tc_fence_before();
  cluster_sync_all();  // the pair's MMAs read both CTAs' memory: nobody leaves early
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, Cfg::kTmemCols);
  }
}

// maps: q, k, v, dO (128-row boxes), dQ accumulator (64-row boxes), q, dO
// (64-row boxes).
cudaError_t launch_attn_bwd_pair_main(const BwdParams& p, const CUtensorMap* maps, int n_pairs,
                                      int* ticket, cudaStream_t st) {
  using Cfg = PairCfg;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int slot = prof_begin(kKBwdMain, st);
  attn_bwd_pair_kernel<<<2 * n_pairs, 512, Cfg::kSmemBytes, st>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], p, ticket);
  e = cudaGetLastError();
  prof_end(slot, st);
  return e;
}

}  // namespace attn

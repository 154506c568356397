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
//             dK  += dS^T Q_i       (TS, dS^T from TMEM)
//             dQ_i = dS K           (SS, dS from shared memory)
//         and adds dQ_i into the fp32 accumulator with vector reductions; in
//         deterministic mode the additions into one query tile happen in
//         ascending key-tile order, enforced by a per-tile semaphore
//         (section 3.2.4).
//   post  dQ = alpha * dQacc -> bf16.
//
// Warp roles of the main kernel (384 threads):
//   warp 0      producer: Q_i and dO_i by TMA into a two-stage ring, LSE_i and D_i
//               (plain loads) into the same stage.
//   warp 1      TMEM owner and MMA issuer (one thread).
//   warps 4-7   "compute": thread r owns key row r: P^T row, dS^T row, and at the
//               end the dK / dV epilogue.
//   warps 8-11  "dQ": thread r owns query row r of the dQ_i tile: TMEM -> registers
//               -> fp32 reductions into the accumulator.
//
// TMEM (512 columns): dV [0, d), dK [d, 2d), S^T / P^T / dS^T [2d, 2d+128),
// dP^T / dQ [2d+128, 2d+256).
#include <cstdint>
#include <cuda_runtime.h>

#include "attn_common.cuh"

namespace attn {

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = kTileM * D * 2;  // one 128-row bf16 tile of Q, dO, K or V
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;             // 2 stages
  static constexpr int kdOOff = kQOff + 2 * kTileBytes;        // 2 stages
  static constexpr int kdSOff = kdOOff + 2 * kTileBytes;       // 128 x 128 bf16
  static constexpr int kStatOff = kdSOff + 128 * 128 * 2;      // per stage: lse2[128], D[128]
  static constexpr int kBarOff = kStatOff + 2 * 2 * 128 * 4;
  static constexpr int kSmemBytes = kBarOff + 256;
  static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128;
  static constexpr uint32_t kTmemCols = 512;
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t qdo_full[2];
  uint64_t qdo_empty[2];
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

__device__ __forceinline__ bool decode_bwd_tile(const BwdParams& p, int idx, BwdTile& t) {
  if (p.cu_seqlens == nullptr) {
    const int nk = (p.N_k + kTileN - 1) / kTileN;
    if (nk == 0) return false;
    t.j = idx % nk;
    const int rest = idx / nk;
    t.h_kv = rest % p.H_kv;
    t.b = rest / p.H_kv;
    if (t.b >= p.B) return false;
    t.row_base = 0;
    t.batch_coord = t.b;
    t.Lq = p.N_q;
    t.Lk = p.N_k;
    t.sem_base = t.b * ((p.N_q + kTileM - 1) / kTileM);
  } else {
    int s = 0, qslots = 0;
    for (; s < p.B; ++s) {
      const int L = p.cu_seqlens[s + 1] - p.cu_seqlens[s];
      const int nk = (L + kTileN - 1) / kTileN;
      if (idx < nk * p.H_kv) break;
      idx -= nk * p.H_kv;
      qslots += (L + kTileM - 1) / kTileM;
    }
    if (s >= p.B) return false;
    const int L = p.cu_seqlens[s + 1] - p.cu_seqlens[s];
    const int nk = (L + kTileN - 1) / kTileN;
    t.j = idx % nk;
    t.h_kv = idx / nk;
    t.b = s;
    t.row_base = p.cu_seqlens[s];
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

// ------------------------------------------------------------------ pre / post

// D[row] = sum_c dO[row, c] * O[row, c]; G = d/16 lanes per (row, head).
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

template <int D>
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

template <int D>
__global__ void __launch_bounds__(384, 1)
attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p, int* ticket) {
  using Cfg = BwdCfg<D>;
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
  if (!decode_bwd_tile(p, bars->work_idx, t)) return;
  const int n_per_head = t.n_qt - t.i_start;
  const int n_it = n_per_head * p.group;
  const long long lim = p.wait_limit;

  if (tid == 0) {
    mbar_init(smem_addr(&bars->kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&bars->qdo_full[s]), 32);
      mbar_init(smem_addr(&bars->qdo_empty[s]), 1);
    }
    mbar_init(smem_addr(&bars->s_full), 1);
    mbar_init(smem_addr(&bars->dp_full), 1);
    mbar_init(smem_addr(&bars->p_ready), 128);
    mbar_init(smem_addr(&bars->ds_ready), 128);
    mbar_init(smem_addr(&bars->dq_full), 1);
    mbar_init(smem_addr(&bars->dq_free), 128);
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

  if (warp < 4) {
    regs_dec<56>();
    if (warp == 0) {
      // ------------------------------------------------------- producer
      if (n_it > 0) {
        if (lane == 0) {
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_do);
          const uint32_t kvb = smem_addr(&bars->kv_full);
          mbar_arrive_expect_tx(kvb, 2 * Cfg::kTileBytes);
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_load_4d(smem_addr(smem + Cfg::kKOff) + hf * 16384, &tm_k, kvb, hf * 64, t.h_kv,
                        t.row_base + t.j * kTileN, t.batch_coord);
            tma_load_4d(smem_addr(smem + Cfg::kVOff) + hf * 16384, &tm_v, kvb, hf * 64, t.h_kv,
                        t.row_base + t.j * kTileN, t.batch_coord);
          }
        }
        float* stat = reinterpret_cast<float*>(smem + Cfg::kStatOff);
        for (int it = 0; it < n_it; ++it) {
          const int stage = it & 1;
          const int h = t.h_kv * p.group + it / n_per_head;
          const int i = t.i_start + it % n_per_head;
          if (!mbar_wait(smem_addr(&bars->qdo_empty[stage]), ((it >> 1) & 1) ^ 1, lim)) {
            record_error(p.err, kErrTimeout);
            break;
          }
          const uint32_t fb = smem_addr(&bars->qdo_full[stage]);
          if (lane == 0) {
            mbar_expect_tx(fb, 2 * Cfg::kTileBytes);
            for (int hf = 0; hf < D / 64; ++hf) {
              tma_load_4d(smem_addr(smem + Cfg::kQOff + stage * Cfg::kTileBytes) + hf * 16384, &tm_q,
                          fb, hf * 64, h, t.row_base + i * kTileM, t.batch_coord);
              tma_load_4d(smem_addr(smem + Cfg::kdOOff + stage * Cfg::kTileBytes) + hf * 16384,
                          &tm_do, fb, hf * 64, h, t.row_base + i * kTileM, t.batch_coord);
            }
          }
          // LSE (to log2 units) and D for the 128 rows of this query tile; rows
          // past the end get LSE = +inf so that their P is exactly 0.
          float* lse2 = stat + stage * 256;
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
          mbar_arrive(fb);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------- MMA issuer
      if (lane == 0 && n_it > 0) {
        constexpr uint32_t kIdSS = make_idesc_bf16(128, 128, 0, 0);     // S^T, dP^T
        constexpr uint32_t kIdTS = make_idesc_bf16(128, D, 0, 1);       // dV, dK
        constexpr uint32_t kIdDQ = make_idesc_bf16(128, D, 1, 1);       // dQ
        const uint32_t k_base = smem_addr(smem + Cfg::kKOff);
        const uint32_t v_base = smem_addr(smem + Cfg::kVOff);
        const uint32_t ds_base = smem_addr(smem + Cfg::kdSOff);
        bool ok = mbar_wait(smem_addr(&bars->kv_full), 0, lim);
        for (int it = 0; ok && it < n_it; ++it) {
          const int stage = it & 1;
          const uint32_t q_base = smem_addr(smem + Cfg::kQOff + stage * Cfg::kTileBytes);
          const uint32_t do_base = smem_addr(smem + Cfg::kdOOff + stage * Cfg::kTileBytes);
          if (!(ok = mbar_wait(smem_addr(&bars->qdo_full[stage]), (it >> 1) & 1, lim))) break;
          tc_fence_after();
          // S^T = K Q^T
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tmem + Cfg::kColS, make_sdesc_sw128(k_base + off, 16, 1024),
                   make_sdesc_sw128(q_base + off, 16, 1024), kIdSS, kk > 0);
          }
          mma_commit(smem_addr(&bars->s_full));
          // dP^T = V dO^T (its TMEM columns hold dQ_{it-1} until that is read out)
          if (it > 0 && !(ok = mbar_wait(smem_addr(&bars->dq_free), (it - 1) & 1, lim))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tmem + Cfg::kColDP, make_sdesc_sw128(v_base + off, 16, 1024),
                   make_sdesc_sw128(do_base + off, 16, 1024), kIdSS, kk > 0);
          }
          mma_commit(smem_addr(&bars->dp_full));
          // dV += P^T dO
          if (!(ok = mbar_wait(smem_addr(&bars->p_ready), it & 1, lim))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            mma_ts(tmem + Cfg::kColDV, tmem + Cfg::kColS + kk * 8,
                   make_sdesc_sw128(do_base + kk * 2048, 16384, 1024), kIdTS, (it > 0 || kk > 0));
          // dK += dS^T Q ; dQ = dS K
          if (!(ok = mbar_wait(smem_addr(&bars->ds_ready), it & 1, lim))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            mma_ts(tmem + Cfg::kColDK, tmem + Cfg::kColS + 64 + kk * 8,
                   make_sdesc_sw128(q_base + kk * 2048, 16384, 1024), kIdTS, (it > 0 || kk > 0));
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ss(tmem + Cfg::kColDP, make_sdesc_sw128(ds_base + kk * 2048, 16384, 1024),
                   make_sdesc_sw128(k_base + kk * 2048, 16384, 1024), kIdDQ, kk > 0);
          mma_commit(smem_addr(&bars->dq_full));
          mma_commit(smem_addr(&bars->qdo_empty[stage]));
        }
        if (!ok) record_error(p.err, kErrTimeout);
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    regs_inc<224>();
    // --------------------------------------------------------- compute (key row r)
    const int r = tid - 128;
    const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
    const int kv = t.j * kTileN + r;       // sequence-relative key row
    const bool kv_ok = kv < t.Lk;
    const float c = p.scale_log2;
    const float* stat = reinterpret_cast<const float*>(smem + Cfg::kStatOff);
    uint8_t* ds_smem = smem + Cfg::kdSOff;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int stage = it & 1;
      const int i = t.i_start + it % n_per_head;
      if (!(ok = mbar_wait(smem_addr(&bars->qdo_full[stage]), (it >> 1) & 1, lim))) break;
      if (!(ok = mbar_wait(smem_addr(&bars->s_full), it & 1, lim))) break;
      tc_fence_after();
      const float* lse2 = stat + stage * 256;
      const float* dvs = lse2 + 128;
      float pr[128];
      {
        uint32_t sr[128];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          tmem_ld32(tmem + lane_base + Cfg::kColS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + cc * 32));
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(sr + cc * 32));
        const bool diag = p.causal && (i == t.j);
#pragma unroll
        for (int q = 0; q < 128; q += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(lse2 + q);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pv = ex2_approx(fmaf(__uint_as_float(sr[q + e]), c, -lv[e]));
            if (diag && (r > q + e)) pv = 0.f;  // key after query: masked
            pr[q + e] = kv_ok ? pv : 0.f;
          }
        }
      }
      {
        uint32_t pk[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) pk[e] = pack_bf16x2(pr[2 * e], pr[2 * e + 1]);
        tmem_st32(tmem + lane_base + Cfg::kColS, *reinterpret_cast<uint32_t(*)[32]>(pk));
        tmem_st32(tmem + lane_base + Cfg::kColS + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_addr(&bars->p_ready));
      // dS^T = P^T o (dP^T - D)
      if (!(ok = mbar_wait(smem_addr(&bars->dp_full), it & 1, lim))) break;
      // the previous dQ MMA read dS from shared memory; it must have finished
      if (it > 0 && !(ok = mbar_wait(smem_addr(&bars->dq_full), (it - 1) & 1, lim))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t dp[32];
        tmem_ld32(tmem + lane_base + Cfg::kColDP + cc * 32, dp);
        tmem_ld_wait(dp);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int q0 = cc * 32 + 2 * e;
          const float d0 = pr[q0] * (__uint_as_float(dp[2 * e]) - dvs[q0]);
          const float d1 = pr[q0 + 1] * (__uint_as_float(dp[2 * e + 1]) - dvs[q0 + 1]);
          w[e] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tmem + lane_base + Cfg::kColS + 64 + cc * 16, w);
        // dS in shared memory as the MN-major A operand of dQ = dS K:
        // block (cc / 2) holds query columns 64 * (cc / 2) ..; row r = key row.
        uint8_t* blk = ds_smem + (cc >> 1) * 16384;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int chunk = (cc & 1) * 4 + ch;  // 16-byte chunk (8 queries) within the 128-byte row
          *reinterpret_cast<uint4*>(blk + sw128_offset(r, chunk)) =
              make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
        }
      }
      tmem_st_wait();
      fence_async_shared();
      tc_fence_before();
      mbar_arrive(smem_addr(&bars->ds_ready));
    }
    if (!ok) record_error(p.err, kErrTimeout);
    // --------------------------------------------------------- dK / dV epilogue
    bool have = ok && n_it > 0;
    if (have) {
      have = mbar_wait(smem_addr(&bars->dq_full), (n_it - 1) & 1, lim);
      if (!have) record_error(p.err, kErrTimeout);
      tc_fence_after();
    }
    {
      // every lane takes part in the (warp-collective) TMEM loads; only rows
      // inside the sequence are stored
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
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t v[32];
          if (have) {
            tmem_ld32(tmem + lane_base + col + cc * 32, v);
            tmem_ld_wait(v);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          if (kv_ok) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[cc * 4 + e] = make_uint4(
                  pack_bf16x2(__uint_as_float(v[8 * e + 0]) * mul, __uint_as_float(v[8 * e + 1]) * mul),
                  pack_bf16x2(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul),
                  pack_bf16x2(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul),
                  pack_bf16x2(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul));
          }
        }
      }
    }
  } else {
    regs_inc<224>();
    // --------------------------------------------------------- dQ (query row r)
    const int r = tid - 256;
    const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int h = t.h_kv * p.group + it / n_per_head;
      const int i = t.i_start + it % n_per_head;
      if (!(ok = mbar_wait(smem_addr(&bars->dq_full), it & 1, lim))) break;
      tc_fence_after();
      uint32_t v[128];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc)
        tmem_ld32(tmem + lane_base + Cfg::kColDP + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(v + cc * 32));
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + cc * 32));
      tc_fence_before();
      mbar_arrive(smem_addr(&bars->dq_free));
      const int q = i * kTileM + r;
      int* sem = nullptr;
      if (p.deterministic) {
        // wait until every key tile before this one has added into query tile i
        sem = p.sem + (static_cast<size_t>(t.sem_base) + i) * p.H_q + h;
        if (r == 0) {
          const long long t0 = clock64();
          while (ld_acquire(sem) != t.j) {
            if (clock64() - t0 > lim) { record_error(p.err, kErrTimeout); break; }
          }
        }
        named_bar_sync(1, 128);
      }
      if (q < t.Lq) {
        const size_t grow = static_cast<size_t>(t.row_base) + q;
        const size_t off = p.cu_seqlens ? (grow * p.H_q + h) * D
                                        : ((static_cast<size_t>(t.b) * p.N_q + q) * p.H_q + h) * D;
        float* dst = p.dq_acc + off;
#pragma unroll
        for (int e = 0; e < D / 4; ++e)
          red_add_v4(dst + 4 * e, __uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                     __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
      }
      if (p.deterministic) {
        __threadfence();
        named_bar_sync(1, 128);
        if (r == 0) atomicAdd(sem, 1);
      }
    }
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

template <int D>
static cudaError_t launch_bwd_impl(const BwdParams& p, const CUtensorMap* maps, cudaStream_t st,
                                   long long rows_q, int n_sem, int n_work) {
  const long long n_rowheads = rows_q * p.H_q;
  const long long n_acc4 = n_rowheads * D / 4;
  const int threads = 256;
  long long want = (n_acc4 + threads - 1) / threads;
  int blocks = static_cast<int>(want < 152 * 16 ? (want > 0 ? want : 1) : 152 * 16);
  int slot = prof_begin(kKBwdPre, st);
  attn_bwd_pre_kernel<D><<<blocks, threads, 0, st>>>(p, n_rowheads, n_acc4, n_sem);
  cudaError_t e = cudaGetLastError();
  prof_end(slot, st);
  if (e != cudaSuccess) return e;
  if (n_work > 0) {
    using Cfg = BwdCfg<D>;
    auto kern = attn_bwd_main_kernel<D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    int* ticket = p.deterministic ? p.sem + n_sem : nullptr;
    slot = prof_begin(kKBwdMain, st);
    kern<<<n_work, 384, Cfg::kSmemBytes, st>>>(maps[0], maps[1], maps[2], maps[3], p, ticket);
    e = cudaGetLastError();
    prof_end(slot, st);
    if (e != cudaSuccess) return e;
  }
  const long long n_vec8 = n_rowheads * D / 8;
  want = (n_vec8 + threads - 1) / threads;
  blocks = static_cast<int>(want < 152 * 16 ? (want > 0 ? want : 1) : 152 * 16);
  slot = prof_begin(kKBwdPost, st);
  attn_bwd_post_kernel<D><<<blocks, threads, 0, st>>>(p, n_vec8);
  e = cudaGetLastError();
  prof_end(slot, st);
  return e;
}

cudaError_t launch_attn_bwd(const BwdParams& p, const CUtensorMap* maps, cudaStream_t stream,
                            long long rows_q, int n_sem, int n_work) {
  if (p.d == 64) return launch_bwd_impl<64>(p, maps, stream, rows_q, n_sem, n_work);
  return launch_bwd_impl<128>(p, maps, stream, rows_q, n_sem, n_work);
}

}  // namespace attn

// Per-row softmax step of the forward kernels (one thread per query row, one
// 128-key S tile): scale, mask, running max with the conditional rescale
// threshold tau, exp2 (MUFU, or partly the FMA-pipe polynomial), row sum and
// the bf16 P row (FlashAttention-4 summary, sections 3.1.3 and 3.1.4).
#pragma once

#include "attn_common.cuh"

namespace attn {

template <int EMU, bool POS_SCALE>
__device__ __forceinline__ void softmax_row_tile(float (&s)[128], float c, float& m_used,
                                                 float& l, int kv0, int qrow, int Lk,
                                                 bool need_mask, int causal,
                                                 uint32_t (&pk)[64], bool& rescale_warp,
                                                 float& factor) {
  if (!POS_SCALE) {
#pragma unroll
    for (int i = 0; i < 128; ++i) s[i] *= c;
  }
  if (need_mask) {
#pragma unroll
    for (int i = 0; i < 128; ++i) {
      const int key = kv0 + i;
      const bool vis = key < Lk && (!causal || key <= qrow);
      s[i] = vis ? s[i] : -INFINITY;
    }
  }
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
  for (int i = 8; i < 128; ++i) mx[i & 7] = fmaxf(mx[i & 7], s[i]);
  float m = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
  if (POS_SCALE) m *= c;  // max of the scaled scores (c > 0)
  const float m_new = fmaxf(m_used, m);
  const bool need = (m_new - m_used) > kTau;  // false when both are -inf (NaN compare)
  rescale_warp = __any_sync(0xffffffffu, need);
  factor = 1.0f;
  if (rescale_warp) {
    if (m_new > m_used) {
      factor = ex2_approx(m_used - m_new);  // 0 when m_used = -inf
      m_used = m_new;
      l *= factor;
    }
  }
  const float mb = (m_used == -INFINITY) ? 0.0f : m_used;
  float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    float x0, x1;
    if (POS_SCALE) {
      x0 = fmaf(s[2 * i], c, -mb);
      x1 = fmaf(s[2 * i + 1], c, -mb);
    } else {
      x0 = s[2 * i] - mb;
      x1 = s[2 * i + 1] - mb;
    }
    float p0, p1;
    if (EMU > 0 && !need_mask && (i & 7) >= 8 - EMU) {
      p0 = exp2_poly3(x0);
      p1 = exp2_poly3(x1);
    } else {
      p0 = ex2_approx(x0);
      p1 = ex2_approx(x1);
    }
    sum[i & 3] += p0 + p1;
    pk[i] = pack_bf16x2(p0, p1);
  }
  l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
}

}  // namespace attn

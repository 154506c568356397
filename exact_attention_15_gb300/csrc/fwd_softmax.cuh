// Per-row softmax step of the forward kernels (one thread per query row, one
// 128-key S tile): scale, mask, running max with the conditional rescale
// threshold tau, exp2 (MUFU, or partly the FMA-pipe polynomial), row sum and
// the bf16 P row (FlashAttention-4 summary, sections 3.1.3 and 3.1.4).
//
// It comes in two phases so that a kernel can hand P to the tensor core in
// parts (section 3.1.2: P is stored in two stages, three quarters and then the
// last quarter): softmax_row_max decides the exponent bias of the tile,
// softmax_row_exp turns a range of packed P words into exponentials.
#pragma once

#include "attn_common.cuh"

namespace attn {

// Scales (unless the scale is folded into the exponent, POS_SCALE) and masks
// the S row, takes its max and applies the conditional rescale rule: the bias
// m_used moves only when the max grew by more than tau for some lane of the
// warp (then every lane of the warp moves to its own max and l is rescaled by
// `factor`, which the caller also applies to O). Returns the bias the
// exponentials subtract (0 for a row that has seen no key yet).
template <bool POS_SCALE>
__device__ __forceinline__ float softmax_row_max(float (&s)[128], float c, float& m_used, float& l,
                                                 int kv0, int qrow, int Lk, bool need_mask,
                                                 int causal, bool& rescale_warp, float& factor) {
  if (!POS_SCALE) {
    const uint64_t c2 = f32x2(c, c);
#pragma unroll
    for (int i = 0; i < 64; ++i) f32x2_split(mul_f32x2(f32x2(s[2 * i], s[2 * i + 1]), c2), s[2 * i], s[2 * i + 1]);
  }
  if (need_mask) {
#pragma unroll
    for (int i = 0; i < 128; ++i) {
      const int key = kv0 + i;
      const bool vis = key < Lk && (!causal || key <= qrow);
      s[i] = vis ? s[i] : -INFINITY;
    }
  }
  // eight independent chains of three-input maxima
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
  for (int i = 16; i < 128; i += 16)
#pragma unroll
    for (int j = 0; j < 8; ++j) mx[j] = max3f(mx[j], s[i + j], s[i + 8 + j]);
  float m = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
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
  return (m_used == -INFINITY) ? 0.0f : m_used;
}

// Packed P words [W0, W1) of the row (word i holds keys 2i and 2i + 1):
// p = 2^(x - mb) with x the scaled score, summed in fp32 before the bf16
// rounding into two packed pair accumulators (sum2[i & 1] adds word i's pair).
// The scale, bias and sum run on packed fp32 pairs, one instruction per key
// pair.
template <int EMU, bool POS_SCALE, int W0, int W1>
__device__ __forceinline__ void softmax_row_exp(const float (&s)[128], float c, float mb,
                                                bool need_mask, uint32_t (&pk)[64],
                                                uint64_t (&sum2)[2]) {
  const uint64_t c2 = f32x2(c, c);
  const uint64_t nb2 = f32x2(-mb, -mb);
#pragma unroll
  for (int i = W0; i < W1; ++i) {
    float x0, x1;
    const uint64_t s2 = f32x2(s[2 * i], s[2 * i + 1]);
    f32x2_split(POS_SCALE ? fma_f32x2(s2, c2, nb2) : add_f32x2(s2, nb2), x0, x1);
    float p0, p1;
    if (EMU > 0 && !need_mask && (i & 7) >= 8 - EMU) {
      exp2_poly3_x2(x0, x1, p0, p1);
    } else {
      p0 = ex2_approx(x0);
      p1 = ex2_approx(x1);
    }
    sum2[i & 1] = add_f32x2(sum2[i & 1], f32x2(p0, p1));
    pk[i] = pack_bf16x2(p0, p1);
  }
}

// Row sum of the two packed pair accumulators.
__device__ __forceinline__ float softmax_row_sum(const uint64_t (&sum2)[2]) {
  float a, b, c, d;
  f32x2_split(sum2[0], a, b);
  f32x2_split(sum2[1], c, d);
  return (a + b) + (c + d);
}

// Both phases over the whole tile, P kept in registers.
template <int EMU, bool POS_SCALE>
__device__ __forceinline__ void softmax_row_tile(float (&s)[128], float c, float& m_used,
                                                 float& l, int kv0, int qrow, int Lk,
                                                 bool need_mask, int causal,
                                                 uint32_t (&pk)[64], bool& rescale_warp,
                                                 float& factor) {
  const float mb = softmax_row_max<POS_SCALE>(s, c, m_used, l, kv0, qrow, Lk, need_mask, causal,
                                              rescale_warp, factor);
  uint64_t sum2[2] = {0ull, 0ull};
  softmax_row_exp<EMU, POS_SCALE, 0, 64>(s, c, mb, need_mask, pk, sum2);
  l += softmax_row_sum(sum2);
}

}  // namespace attn

// Warp-per-token biased top-k and gates, shared by both router paths.
//
// Lesson "Mixture of Experts", "Build it" step 1: the bias is added to a token's scores
// only to choose its experts (descending order, ties to the lower id); the gates are a
// softmax over the chosen experts' original scores.  The sigmoid and sqrt(softplus)
// routers read the same way with s = sigmoid(logit) or s = sqrt(ln(1 + e^logit)):
// selection on s + bias, gates s_j / sum of the chosen s.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// score function codes (as moe_score_fn_t)
enum : int { kScoreSoftmax = 0, kScoreSigmoid = 1, kScoreSqrtSoftplus = 2 };

// Unbiased score s of a logit for the sigmoid / sqrt(softplus) routers.
__device__ __forceinline__ float router_score(float l, int fn) {
  if (fn == kScoreSigmoid) return 1.0f / (1.0f + expf(-l));
  const float sp = fmaxf(l, 0.0f) + log1pf(expf(-fabsf(l)));  // softplus without overflow
  return sqrtf(sp);
}

// lg[i] = logit of expert lane + 32 i for this warp's token (entries with id >= E ignored).
// Lane j < k writes idx_row[j] / gate_row[j]; lane 0 writes *tie_out (if non-null).  A NaN or
// infinite logit (the gates are then undefined) sets kStatusNonFiniteLogit in *status; the
// selection still follows the order rule (NaN scores last).
template <int PER>
__device__ __forceinline__ void warp_topk_gates(const float (&lg)[PER], int lane, int E, int k,
                                                const float* __restrict__ bias, int score_fn,
                                                int32_t* __restrict__ idx_row, float* __restrict__ gate_row,
                                                uint8_t* __restrict__ tie_out, int* __restrict__ status) {
  bool nonfinite = false;
#pragma unroll
  for (int i = 0; i < PER; ++i) nonfinite |= (lane + 32 * i < E) && !isfinite(lg[i]);
  if (__any_sync(0xffffffffu, nonfinite) && lane == 0) atomicOr(status, kStatusNonFiniteLogit);
  float v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    float key = -INFINITY;
    if (e < E) {
      const float sc = score_fn == kScoreSoftmax ? lg[i] : router_score(lg[i], score_fn);
      const float sl = sc + (bias ? bias[e] : 0.0f);
      key = isnan(sl) ? -INFINITY : sl;
    }
    v[i] = key;
  }
  // Each round: every lane offers its best untaken (key, id); one warp max-reduction over
  // an order-preserving integer image of the key, then one min-reduction over the ids of
  // the lanes holding that key, pick the winner (key desc, id asc) in two instructions.
  uint32_t ord[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const uint32_t u = __float_as_uint(v[i] + 0.0f);  // -0 -> +0: equal keys stay equal
    ord[i] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  uint32_t taken = 0;
  int my_id = 0;
  float my_lg = 0.f, kth = 0.f, next = -INFINITY;
  const int rounds = k < E ? k + 1 : k;
  for (int r = 0; r < rounds; ++r) {
    uint32_t bo = 0u, bi = 0xffffffffu;
    int bslot = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {  // ids grow with i: the first maximum has the lowest id
      const bool free = !((taken >> i) & 1u);
      if (free && (bi == 0xffffffffu || ord[i] > bo)) { bo = ord[i]; bi = (uint32_t)(lane + 32 * i); bslot = i; }
    }
    const uint32_t wo = __reduce_max_sync(0xffffffffu, bo);
    const uint32_t wi = __reduce_min_sync(0xffffffffu, (bi != 0xffffffffu && bo == wo) ? bi : 0xffffffffu);
    const int owner = (int)(wi & 31u), slot = (int)(wi >> 5);
    const uint32_t wu = (wo & 0x80000000u) ? (wo & 0x7fffffffu) : ~wo;  // back to float bits
    const float bv = __uint_as_float(wu);
    if (r < k) {
      float cand = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (i == slot) cand = lg[i];
      const float wl = __shfl_sync(0xffffffffu, cand, owner);
      if (lane == r) { my_id = (int)wi; my_lg = wl; }
      if (owner == lane) taken |= 1u << slot;
      if (r == k - 1) kth = bv;
    } else {
      next = bv;
    }
    (void)bslot;
  }
  const bool act = lane < k;
  float g;
  if (score_fn != kScoreSoftmax) {
    const float s = act ? router_score(my_lg, score_fn) : 0.f;
    float sum = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    g = s / sum;
  } else {
    float m = act ? my_lg : -INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float ex = act ? expf(my_lg - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    g = ex / sum;
  }
  if (act) {
    idx_row[lane] = my_id;
    gate_row[lane] = g;
  }
  if (tie_out && lane == 0) *tie_out = (k < E && (kth - next) < 1e-6f) ? 1 : 0;
}

}  // namespace moe

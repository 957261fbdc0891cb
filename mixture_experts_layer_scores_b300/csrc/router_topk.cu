// Router GEMM + score function + biased top-k + gates, one fused kernel.
//
// Lesson "Mixture of Experts" (AI Engineering from Scratch), "Build it" step 1:
// raw dot-product scores, bias added for selection only, stable descending order,
// gates from the chosen experts' original scores.  Handbook article, router-precision
// paragraph: the router stays in fp32.
//
// Each block scores 32 tokens against all E (<= 256) experts on CUDA cores in fp32.
// Every output accumulates 32-element partial sums with FMA and folds them into a
// running total with a two-sum (error-free) addition, so the logits sit within a few
// 1e-8 of the correctly rounded dot product.  The 32 x E logit tile then stays in
// shared memory for a warp-per-token top-k: each lane holds E/32 scores in registers
// and k+1 rounds of a shuffle arg-max (score desc, id asc) pick the experts and the
// (k+1)-th score for the near-tie flag.
#include "topk_common.cuh"

namespace moe {
namespace {

constexpr int BT = 32;   // tokens per block
constexpr int BK = 32;   // reduction chunk
constexpr int NT = 256;  // threads per block

template <typename XT>
struct XLoad;

template <>
struct XLoad<__nv_bfloat16> {
  // 32 tokens x 32 bf16 = 128 vectors of 16 B; threads 0..127 take one each.
  uint4 v;
  __device__ void load(const __nv_bfloat16* x, int N, int D, int n0, int k0, int t) {
    v = make_uint4(0, 0, 0, 0);
    if (t < 128) {
      int n = n0 + (t >> 2), q = t & 3;
      if (n < N) v = *reinterpret_cast<const uint4*>(x + (size_t)n * D + k0 + q * 8);
    }
  }
  __device__ void store(float* xs, int t) {
    if (t < 128) {
      float f[8];
      bf16x8_to_f32(v, f);
      int n = t >> 2, q = t & 3;
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[(q * 8 + i) * BT + n] = f[i];
    }
  }
};

template <>
struct XLoad<float> {
  // 32 tokens x 32 fp32 = 256 vectors of 16 B; one per thread.
  float4 v;
  __device__ void load(const float* x, int N, int D, int n0, int k0, int t) {
    v = make_float4(0.f, 0.f, 0.f, 0.f);
    int n = n0 + (t >> 3), q = t & 7;
    if (n < N) v = *reinterpret_cast<const float4*>(x + (size_t)n * D + k0 + q * 4);
  }
  __device__ void store(float* xs, int t) {
    int n = t >> 3, q = t & 7;
    xs[(q * 4 + 0) * BT + n] = v.x;
    xs[(q * 4 + 1) * BT + n] = v.y;
    xs[(q * 4 + 2) * BT + n] = v.z;
    xs[(q * 4 + 3) * BT + n] = v.w;
  }
};

template <int EP>
struct WLoad {
  // EP rows x 32 fp32 = EP*8 vectors; LPR threads share a row.
  static constexpr int LPR = NT / EP;
  static constexpr int VPT = 8 / LPR;
  float4 v[VPT];
  __device__ void load(const float* w, int E, int D, int k0, int t) {
    int e = t / LPR, part = t % LPR;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < E) v[i] = *reinterpret_cast<const float4*>(w + (size_t)e * D + k0 + (part * VPT + i) * 4);
    }
  }
  __device__ void store(float* ws, int t) {
    int e = t / LPR, part = t % LPR;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      int kk = (part * VPT + i) * 4;
      ws[(kk + 0) * EP + e] = v[i].x;
      ws[(kk + 1) * EP + e] = v[i].y;
      ws[(kk + 2) * EP + e] = v[i].z;
      ws[(kk + 3) * EP + e] = v[i].w;
    }
  }
};

template <typename XT, int EP, int TM, int TE>
__global__ void __launch_bounds__(NT) router_topk_kernel(
    const XT* __restrict__ xn, const float* __restrict__ w, const float* __restrict__ bias,
    int N, int D, int E, int k, int score_fn, float* __restrict__ logits_out,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate, uint8_t* __restrict__ near_tie,
    int* __restrict__ status) {
  constexpr int TGE = EP / TE;  // threads along experts
  static_assert(TGE * (BT / TM) == NT, "thread tile");
  extern __shared__ __align__(16) float smem[];
  float* xs = smem;                 // [2][BK][BT]
  float* ws = smem + 2 * BK * BT;   // [2][BK][EP]

  const int t = threadIdx.x;
  const int te = t % TGE, tm = t / TGE;
  const int n0 = blockIdx.x * BT;
  grid_dep_wait();
  grid_dep_launch();

  float acc_s[TM][TE], acc_c[TM][TE];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc_s[i][j] = acc_c[i][j] = 0.f;

  XLoad<XT> xl;
  WLoad<EP> wl;
  xl.load(xn, N, D, n0, 0, t);
  wl.load(w, E, D, 0, t);
  xl.store(xs, t);
  wl.store(ws, t);

  const int nk = D / BK;
  for (int kc = 0; kc < nk; ++kc) {
    const int buf = kc & 1;
    __syncthreads();
    if (kc + 1 < nk) {
      xl.load(xn, N, D, n0, (kc + 1) * BK, t);
      wl.load(w, E, D, (kc + 1) * BK, t);
    }
    const float* xb = xs + buf * BK * BT;
    const float* wb = ws + buf * BK * EP;
    float p[TM][TE];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TE; ++j) p[i][j] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[TM], b[TE];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = xb[kk * BT + tm * TM + i];
#pragma unroll
      for (int j = 0; j < TE; ++j) b[j] = wb[kk * EP + te * TE + j];
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TE; ++j) p[i][j] = fmaf(a[i], b[j], p[i][j]);
    }
    // two-sum: fold the chunk partial into the running total without losing its error
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TE; ++j) {
        float s = acc_s[i][j], q = p[i][j];
        float tt = s + q;
        float bp = tt - s;
        float err = (s - (tt - bp)) + (q - bp);
        acc_s[i][j] = tt;
        acc_c[i][j] += err;
      }
    if (kc + 1 < nk) {
      xl.store(xs + (buf ^ 1) * BK * BT, t);
      wl.store(ws + (buf ^ 1) * BK * EP, t);
    }
  }
  __syncthreads();

  // logit tile -> shared memory (reusing the weight buffers) and, optionally, global
  float* lt = ws;  // [BT][EP + 1]
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int nl = tm * TM + i, n = n0 + nl;
#pragma unroll
    for (int j = 0; j < TE; ++j) {
      const int e = te * TE + j;
      const float v = acc_s[i][j] + acc_c[i][j];
      lt[nl * (EP + 1) + e] = v;
      if (logits_out && n < N && e < E) logits_out[(size_t)n * E + e] = v;
    }
  }
  __syncthreads();

  // warp-per-token top-k
  const int lane = t & 31, warp = t >> 5;
  constexpr int PER = EP / 32;
  for (int nl = warp; nl < BT; nl += NT / 32) {
    const int n = n0 + nl;
    if (n >= N) break;
    float lg[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) lg[i] = lt[nl * (EP + 1) + lane + 32 * i];
    warp_topk_gates<PER>(lg, lane, E, k, bias, score_fn, topk_idx + (size_t)n * k,
                         topk_gate + (size_t)n * k, near_tie ? near_tie + n : nullptr, status);
  }
}

template <typename XT, int EP, int TM, int TE>
moe_status_t launch(const void* xn, int N, int D, const float* w, const float* bias, int E, int k,
                    int score_fn, float* logits, int32_t* idx, float* gate, uint8_t* tie, int* status,
                    cudaStream_t s) {
  const size_t smem = (size_t)(2 * BK * BT + 2 * BK * EP) * sizeof(float);
  auto kern = router_topk_kernel<XT, EP, TM, TE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int grid = (N + BT - 1) / BT;
  return launch_kernel(kern, dim3(grid), dim3(NT), smem, s, static_cast<const XT*>(xn), w, bias, N, D, E, k,
                       score_fn, logits, idx, gate, tie, status);
}

template <typename XT>
moe_status_t dispatch(const void* xn, int N, int D, const float* w, const float* bias, int E, int k,
                      int score_fn, float* logits, int32_t* idx, float* gate, uint8_t* tie, int* status,
                      cudaStream_t s) {
  if (E <= 32) return launch<XT, 32, 2, 2>(xn, N, D, w, bias, E, k, score_fn, logits, idx, gate, tie, status, s);
  if (E <= 64) return launch<XT, 64, 2, 4>(xn, N, D, w, bias, E, k, score_fn, logits, idx, gate, tie, status, s);
  if (E <= 128) return launch<XT, 128, 4, 4>(xn, N, D, w, bias, E, k, score_fn, logits, idx, gate, tie, status, s);
  return launch<XT, 256, 4, 8>(xn, N, D, w, bias, E, k, score_fn, logits, idx, gate, tie, status, s);
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_router_topk(const void* xn, moe_dtype_t x_dtype, int N, int D,
                                        const float* w_router, const float* bias, int E, int k,
                                        moe_score_fn_t fn, float* logits_out, int32_t* topk_idx,
                                        float* topk_gate, uint8_t* near_tie, moe_stream_t stream) {
  using namespace moe;
  if (N < 0 || D <= 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > MOE_MAX_EXPERTS_CUDA_CORE || k > MOE_MAX_TOPK || D % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (fn != MOE_SCORE_SOFTMAX && fn != MOE_SCORE_SIGMOID && fn != MOE_SCORE_SQRT_SOFTPLUS) return MOE_ERR_INVALID_ARG;
  if (x_dtype != MOE_BF16 && x_dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (!xn || !w_router || !topk_idx || !topk_gate) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xn) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  const int sig = (int)fn;  // score function code
  int* status = device_status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = as_cuda(stream);
  if (x_dtype == MOE_BF16)
    return dispatch<__nv_bfloat16>(xn, N, D, w_router, bias, E, k, sig, logits_out, topk_idx,
                                   topk_gate, near_tie, status, s);
  return dispatch<float>(xn, N, D, w_router, bias, E, k, sig, logits_out, topk_idx, topk_gate,
                         near_tie, status, s);
}

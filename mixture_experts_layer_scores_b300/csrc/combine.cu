// Un-permute + gate-weighted combine, and the +-gamma bias step.
//
// Lesson "Mixture of Experts", section "Concept": out = h + sum_j gate_j * Expert_j(x),
// "Shared experts": the always-on expert adds its output with weight 1.
// "Load-balancing problem" item 3 and "Build it" step 2: each expert's bias moves by
// gamma against the sign of its load error.
#include "moe_internal.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

template <typename T>
struct Vec;  // one 16-byte vector of T as floats

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int W = 8;
  __device__ static void load(const void* p, float* f) {
    bf16x8_to_f32(__ldg(static_cast<const uint4*>(p)), f);
  }
  __device__ static void load_shared(const void* p, float* f) {
    bf16x8_to_f32(*static_cast<const uint4*>(p), f);
  }
  __device__ static void store(void* p, const float* f) {
    *static_cast<uint4*>(p) = f32_to_bf16x8(f);
  }
};

template <>
struct Vec<float> {
  static constexpr int W = 4;
  __device__ static void load(const void* p, float* f) {
    const float4 v = __ldg(static_cast<const float4*>(p));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ static void load_shared(const void* p, float* f) {
    const float4 v = *static_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ static void store(void* p, const float* f) {
    *static_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

// One CTA per (TPC tokens, column chunk of CHB bytes); thread i owns the chunk's 16-byte
// vector i of each of its tokens.  Each thread starts async copies (cp.async, L2 only) of its
// vectors from every token's k expert rows and its shared-expert and residual rows into shared
// memory, waits for its own copies, then weights and sums them in slot order and writes out.
// The copies keep TPC * (k + 2) loads per thread in flight without holding registers for them;
// TPC grows for small k (k = 2: two tokens, eight copies) so that a CTA's one round trip for
// its tokens' row indices and gates is shared by enough data loads.  A loop of dependent
// register loads over j does not keep HBM busy.
constexpr int CHB = 2048;
constexpr int THREADS = CHB / 16;

// tokens per CTA for k experts per token: at least ~8 copies in flight per thread
inline int tokens_per_cta(int k) { return k >= 6 ? 1 : (8 + k + 1) / (k + 2); }

template <typename T>
__global__ void __launch_bounds__(THREADS) combine_kernel(const T* __restrict__ y, const int32_t* __restrict__ row_map,
                                                          const float* __restrict__ gate, int N, int k, int D,
                                                          int tpc, const T* __restrict__ shared_y,
                                                          const T* __restrict__ residual, T* __restrict__ out) {
  using namespace tc;
  constexpr int W = Vec<T>::W;
  extern __shared__ __align__(16) uint8_t stage[];  // [tpc][k + 2][CHB]: expert rows, shared, residual
  __shared__ int rows[4 * MOE_MAX_TOPK];
  __shared__ float gs[4 * MOE_MAX_TOPK];
  const int rowbytes = D * (int)sizeof(T);
  const int nch = (rowbytes + CHB - 1) / CHB;
  const int n0 = (blockIdx.x / nch) * tpc, c = blockIdx.x % nch;
  const int nt = min(tpc, N - n0);  // tokens of this CTA
  grid_dep_wait();
  grid_dep_launch();
  if (threadIdx.x < nt * k) {
    rows[threadIdx.x] = row_map[(size_t)n0 * k + threadIdx.x];
    gs[threadIdx.x] = gate[(size_t)n0 * k + threadIdx.x];
  }
  __syncthreads();
  const int off = c * CHB + threadIdx.x * 16;
  if (off >= rowbytes) return;
  const int per = (k + 2) * CHB;  // shared-memory bytes of one token
  const uint32_t mine = smem_u32(stage) + threadIdx.x * 16;
  const uint8_t* yb = reinterpret_cast<const uint8_t*>(y);
  for (int t = 0; t < nt; ++t) {
    const int n = n0 + t;
    for (int j = 0; j < k; ++j)
      if (rows[t * k + j] >= 0) cp_async_16(mine + t * per + j * CHB, yb + (size_t)rows[t * k + j] * rowbytes + off, 16);
    if (shared_y)
      cp_async_16(mine + t * per + k * CHB, reinterpret_cast<const uint8_t*>(shared_y) + (size_t)n * rowbytes + off,
                  16);
    if (residual)
      cp_async_16(mine + t * per + (k + 1) * CHB,
                  reinterpret_cast<const uint8_t*>(residual) + (size_t)n * rowbytes + off, 16);
  }
  cp_async_commit();
  cp_async_wait<0>();
  for (int t = 0; t < nt; ++t) {
    const uint8_t* v = stage + t * per + threadIdx.x * 16;
    float acc[W];
#pragma unroll
    for (int i = 0; i < W; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      if (rows[t * k + j] < 0) continue;  // dropped slot
      float f[W];
      Vec<T>::load_shared(v + j * CHB, f);
      const float g = gs[t * k + j];
#pragma unroll
      for (int i = 0; i < W; ++i) acc[i] = fmaf(g, f[i], acc[i]);
    }
    if (shared_y) {
      float f[W];
      Vec<T>::load_shared(v + k * CHB, f);
#pragma unroll
      for (int i = 0; i < W; ++i) acc[i] += f[i];
    }
    if (residual) {
      float f[W];
      Vec<T>::load_shared(v + (k + 1) * CHB, f);
#pragma unroll
      for (int i = 0; i < W; ++i) acc[i] += f[i];
    }
    Vec<T>::store(reinterpret_cast<uint8_t*>(out) + (size_t)(n0 + t) * rowbytes + off, acc);
  }
}

__global__ void bias_update_kernel(const int32_t* __restrict__ counts, int E, long long total,
                                   float gamma, float* __restrict__ bias, float* __restrict__ mom) {
  __shared__ int smax[32];
  grid_dep_wait();
  grid_dep_launch();
  int m = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const long long c = counts[e];
    const long long d = total - (long long)E * c;  // sign(total/E - c), exactly
    const float sg = d > 0 ? 1.f : (d < 0 ? -1.f : 0.f);
    bias[e] = bias[e] + gamma * sg;
    m = max(m, (int)c);
  }
  if (mom) {
    for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      int mm = 0;
      for (int w = 0; w < (int)(blockDim.x + 31) / 32; ++w) mm = max(mm, smax[w]);
      *mom = total > 0 ? (float)((double)mm * E / (double)total) : 0.f;
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_unpermute_combine(const void* y_perm, const int32_t* row_map,
                                              const float* topk_gate, int N, int k, int D,
                                              const void* shared_y, const void* residual, void* out,
                                              moe_dtype_t dtype, moe_stream_t stream) {
  using namespace moe;
  if (N < 0 || k < 1 || D <= 0) return MOE_ERR_INVALID_ARG;
  if (k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  const int esize = dtype == MOE_BF16 ? 2 : 4;
  if ((D * esize) % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (!y_perm || !row_map || !topk_gate || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out) || (shared_y && !aligned16(shared_y)) ||
      (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  const int tpc = tokens_per_cta(k);
  const long long blocks = (long long)((N + tpc - 1) / tpc) * ((D * esize + CHB - 1) / CHB);
  if (blocks > 0x7fffffffll) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = as_cuda(stream);
  const size_t smem = (size_t)tpc * (k + 2) * CHB;  // at most 36 KB: no opt-in needed
  if (dtype == MOE_BF16)
    return launch_kernel(combine_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(THREADS), smem, s,
                         static_cast<const __nv_bfloat16*>(y_perm), row_map, topk_gate, N, k, D, tpc,
                         static_cast<const __nv_bfloat16*>(shared_y), static_cast<const __nv_bfloat16*>(residual),
                         static_cast<__nv_bfloat16*>(out));
  return launch_kernel(combine_kernel<float>, dim3((unsigned)blocks), dim3(THREADS), smem, s,
                       static_cast<const float*>(y_perm), row_map, topk_gate, N, k, D, tpc,
                       static_cast<const float*>(shared_y), static_cast<const float*>(residual),
                       static_cast<float*>(out));
}

extern "C" moe_status_t moe_bias_update(const int32_t* counts, int E, int64_t total_assignments,
                                        float gamma, float* bias, float* max_over_mean_out,
                                        moe_stream_t stream) {
  using namespace moe;
  if (E < 1 || total_assignments < 0 || !counts || !bias) return MOE_ERR_INVALID_ARG;
  if (E > 1 << 20) return MOE_ERR_UNSUPPORTED;
  return launch_kernel(bias_update_kernel, dim3(1), dim3(1024), 0, as_cuda(stream), counts, E,
                       (long long)total_assignments, gamma, bias, max_over_mean_out);
}

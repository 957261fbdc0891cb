// Per-expert histogram, exclusive scan and stable permutation of routed rows.
//
// Lesson "Mixture of Experts", "Build it" step 2 (count how often each expert fires)
// and the evaluation article's per-expert routed-token histogram.  The permutation
// lays each expert's tokens out as one contiguous block of rows so the grouped GEMM
// reads them with TMA; within an expert, rows follow slot order n*k + j (stable).
//
// Deterministic, no order-dependent atomics:
//   1. hist : block b counts the ids of its slot chunk in shared memory -> ws[b][E]
//   2. scan : one block turns ws into per-chunk positions (slots of expert e in earlier
//             chunks), writes counts (the routed demand) and offsets (exclusive scan of
//             the kept counts min(count, capacity)) and, when asked, applies the +-gamma
//             bias step to those counts (moe_permute_update_bias)
//   3. rank : block b walks its chunk in slot order; __match_any_sync gives each slot
//             its rank among same-expert slots of the warp, a per-warp table orders the
//             warps; position = chunk position + rank, row = offsets[e] + position while
//             position < capacity, else -1 (dropped).  Writes row_map and perm_token.
//   4. copy : grid-stride 16-byte row moves xn[n] -> x_perm[row_map[n, j]], each source
//             vector read once and written k times.
#include <cmath>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kChunkBlocks = 128;  // target number of slot chunks

struct Plan {
  int tpb;  // tokens per chunk
  int nb;   // number of chunks
};

Plan plan(int N) {
  Plan p;
  p.tpb = (N + kChunkBlocks - 1) / kChunkBlocks;
  if (p.tpb < 1) p.tpb = 1;
  p.nb = (N + p.tpb - 1) / p.tpb;
  return p;
}

__global__ void __launch_bounds__(256) hist_kernel(const int32_t* __restrict__ idx, int R, int E,
                                                   int C, int32_t* __restrict__ ws,
                                                   int* __restrict__ status) {
  extern __shared__ int sh[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  grid_dep_wait();
  grid_dep_launch();
  __syncthreads();
  const int s0 = blockIdx.x * C, s1 = min(R, s0 + C);
  bool bad = false;
  for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
    const int e = idx[s];
    if (e >= 0 && e < E) atomicAdd(&sh[e], 1);
    else bad = true;
  }
  if (bad) atomicOr(status, kStatusBadExpertId);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) ws[(size_t)blockIdx.x * E + e] = sh[e];
}

// The +-gamma step on this call's counts (lesson "Load-balancing problem" item 3):
// bias[e] += gamma * sign(total/E - c_e), the sign taken exactly on integers; and the
// max/mean load.  Called by every thread of one block with the block's counts in `cnt`.
__device__ __forceinline__ void bias_step_block(const int* cnt, int E, long long total, float gamma,
                                                float* __restrict__ bias, float* __restrict__ mom, int* red) {
  int m = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const long long c = cnt[e];
    const long long d = total - (long long)E * c;
    const float sg = d > 0 ? 1.f : (d < 0 ? -1.f : 0.f);
    if (bias) bias[e] = bias[e] + gamma * sg;
    m = max(m, (int)c);
  }
  if (!mom) return;
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    int mm = 0;
    for (int w = 0; w < (int)(blockDim.x + 31) / 32; ++w) mm = max(mm, red[w]);
    *mom = total > 0 ? (float)((double)mm * E / (double)total) : 0.f;
  }
}

// One block of 1024 threads, E <= 1024.  Thread (g, e) owns expert e over chunk range g.
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ ws, int nb, int E, int capacity,
                                                    int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets, long long total, float gamma,
                                                    float* __restrict__ bias, float* __restrict__ mom) {
  extern __shared__ int sh[];  // part[P][E], cnt[E], wsum[32]
  const int P = blockDim.x / E;
  int* part = sh;
  int* cnt = sh + P * E;
  int* wsum = cnt + E;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int g = t / E, e = t % E;
  const int per = (nb + P - 1) / P;
  const int b0 = g * per, b1 = min(nb, b0 + per);
  grid_dep_wait();
  grid_dep_launch();
  if (g < P) {
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += ws[(size_t)b * E + e];
    part[g * E + e] = sum;
  }
  __syncthreads();
  if (t < E) {  // exclusive prefix over chunk groups, per expert
    int c = 0;
    for (int gg = 0; gg < P; ++gg) {
      const int v = part[gg * E + t];
      part[gg * E + t] = c;
      c += v;
    }
    cnt[t] = c;
  }
  __syncthreads();
  // block-wide exclusive scan of the kept counts min(cnt, capacity)
  const int demand = t < E ? cnt[t] : 0;
  const int mine = min(demand, capacity);
  int v = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += y;
  }
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  const int excl = v - mine + (warp > 0 ? wsum[warp - 1] : 0);
  if (t < E) {
    counts[t] = demand;
    offsets[t] = excl;
    if (t == E - 1) offsets[E] = excl + mine;
  }
  if (g < P) {  // position of chunk b's first slot of expert e within the expert
    int base = part[g * E + e];
    for (int b = b0; b < b1; ++b) {
      const int x = ws[(size_t)b * E + e];
      ws[(size_t)b * E + e] = base;
      base += x;
    }
  }
  if (bias || mom) {  // the +-gamma step on these counts (every thread of the block)
    __syncthreads();
    bias_step_block(cnt, E, total, gamma, bias, mom, wsum);
  }
}

__global__ void __launch_bounds__(256) rank_kernel(const int32_t* __restrict__ idx, int R, int k,
                                                   int E, int C, int capacity, const int32_t* __restrict__ ws,
                                                   const int32_t* __restrict__ offsets,
                                                   int32_t* __restrict__ row_map,
                                                   int32_t* __restrict__ perm_token) {
  extern __shared__ int sh[];
  int* running = sh;          // [E]
  int* wcnt = sh + E;         // [8][E]
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  grid_dep_wait();
  grid_dep_launch();
  for (int e = t; e < E; e += 256) {
    running[e] = ws[(size_t)blockIdx.x * E + e];
#pragma unroll
    for (int w = 0; w < 8; ++w) wcnt[w * E + e] = 0;
  }
  __syncthreads();
  const int s0 = blockIdx.x * C, s1 = min(R, s0 + C);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = s0; base < s1; base += 256) {
    const int s = base + t;
    int e = -1;
    if (s < s1) {
      e = idx[s];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += wcnt[w * E + e];
      const int pos = running[e] + pre + rank;
      if (pos < capacity) {
        const int row = offsets[e] + pos;
        row_map[s] = row;
        perm_token[row] = s / k;
      } else {
        row_map[s] = -1;  // over capacity: this slot skips the expert
      }
    } else if (s < s1) {
      row_map[s] = -1;
    }
    __syncthreads();
    for (int x = t; x < E; x += 256) {
      int sum = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        sum += wcnt[w * E + x];
        wcnt[w * E + x] = 0;
      }
      running[x] += sum;
    }
    __syncthreads();
  }
}

// x_perm[row_map[n, j]] = xn[n] in 16-byte vectors; V vectors per row.
__global__ void __launch_bounds__(256) copy_kernel(const uint4* __restrict__ xn, int N, int V, int k,
                                                   const int32_t* __restrict__ row_map,
                                                   uint4* __restrict__ x_perm) {
  constexpr int U = 4;
  grid_dep_wait();
  grid_dep_launch();
  const long long total = (long long)N * V;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += stride * U) {
    uint4 v[U];
    long long it[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      it[u] = i0 + u * stride;
      if (it[u] < total) v[u] = __ldg(xn + it[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (it[u] >= total) continue;
      const int n = (int)(it[u] / V), c = (int)(it[u] % V);
      for (int j = 0; j < k; ++j) {
        const int row = __ldg(row_map + (size_t)n * k + j);
        if (row >= 0) x_perm[(size_t)row * V + c] = v[u];
      }
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_permute_workspace_bytes(int N, int k, int E) {
  if (N <= 0 || k <= 0 || E <= 0) return 0;
  const moe::Plan p = moe::plan(N);
  return (size_t)p.nb * (size_t)E * sizeof(int32_t);
}

extern "C" int64_t moe_expert_capacity(double capacity_factor, int N, int k, int E) {
  if (!(capacity_factor >= 0.0) || N < 0 || k < 1 || E < 1) return -1;
  // evaluated left to right in double, like ceil(C * N * k / E) written out
  const double slots = std::ceil(capacity_factor * (double)N * (double)k / (double)E);
  const int64_t all = (int64_t)N * k;
  return slots >= (double)all ? all : (int64_t)slots;
}

namespace moe {
namespace {

// Every permute entry point: histogram, scan, ranks, and the row copy when x_perm is given;
// with `bias` or `mom`, the +-gamma step on this call's counts as well.
moe_status_t permute_impl(const void* xn, moe_dtype_t dtype, int N, int D, const int32_t* topk_idx, int k, int E,
                          int capacity, int32_t* counts, int32_t* offsets, int32_t* row_map, int32_t* perm_token,
                          void* x_perm, void* workspace, size_t workspace_bytes, float gamma, float* bias,
                          float* mom, cudaStream_t s) {
  if (N < 0 || k < 1 || E < 1 || k > E || D <= 0 || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || (long long)N * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if ((row_map == nullptr) != (perm_token == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x_perm && (!row_map || !xn)) return MOE_ERR_INVALID_ARG;
  if (N == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (bias || mom) return moe_bias_update(counts, E, 0, gamma, bias, mom, reinterpret_cast<moe_stream_t>(s));
    return MOE_OK;
  }
  if (!topk_idx || !workspace) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_permute_workspace_bytes(N, k, E)) return MOE_ERR_INVALID_ARG;
  const size_t esize = dtype == MOE_BF16 ? 2 : 4;
  if (x_perm && ((D * esize) % 16 != 0 || !aligned16(xn) || !aligned16(x_perm)))
    return MOE_ERR_INVALID_ARG;
  int* status = device_status_word();
  if (!status) return MOE_ERR_CUDA;

  const Plan p = plan(N);
  const int R = N * k, C = p.tpb * k;
  int32_t* ws = static_cast<int32_t*>(workspace);
  moe_status_t st = launch_kernel(hist_kernel, dim3(p.nb), dim3(256), E * sizeof(int), s, topk_idx, R, E, C, ws,
                                  status);
  if (st != MOE_OK) return st;
  const int P = 1024 / E;
  st = launch_kernel(scan_kernel, dim3(1), dim3(1024), (size_t)(P * E + E + 32) * sizeof(int), s, ws, p.nb, E,
                     capacity, counts, offsets, (long long)R, gamma, bias, mom);
  if (st != MOE_OK) return st;
  if (row_map) {
    st = launch_kernel(rank_kernel, dim3(p.nb), dim3(256), (size_t)9 * E * sizeof(int), s, topk_idx, R, k, E, C,
                       capacity, static_cast<const int32_t*>(ws), static_cast<const int32_t*>(offsets), row_map,
                       perm_token);
    if (st != MOE_OK) return st;
  }
  if (x_perm) {
    const int V = (int)(D * esize / 16);
    long long items = (long long)N * V;
    long long blocks = (items + 256 * 4 - 1) / (256 * 4);
    const long long cap = (long long)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return launch_kernel(copy_kernel, dim3((unsigned)blocks), dim3(256), 0, s, static_cast<const uint4*>(xn), N, V, k,
                         static_cast<const int32_t*>(row_map), static_cast<uint4*>(x_perm));
  }
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_capacity(const void* xn, moe_dtype_t dtype, int N, int D,
                                             const int32_t* topk_idx, int k, int E, int capacity,
                                             int32_t* counts, int32_t* offsets, int32_t* row_map,
                                             int32_t* perm_token, void* x_perm, void* workspace,
                                             size_t workspace_bytes, moe_stream_t stream) {
  return moe::permute_impl(xn, dtype, N, D, topk_idx, k, E, capacity, counts, offsets, row_map, perm_token, x_perm,
                           workspace, workspace_bytes, 0.f, nullptr, nullptr, moe::as_cuda(stream));
}

extern "C" moe_status_t moe_permute_update_bias(const void* xn, moe_dtype_t dtype, int N, int D,
                                                const int32_t* topk_idx, int k, int E, int capacity,
                                                int32_t* counts, int32_t* offsets, int32_t* row_map,
                                                int32_t* perm_token, void* x_perm, void* workspace,
                                                size_t workspace_bytes, float gamma, float* bias,
                                                float* max_over_mean_out, moe_stream_t stream) {
  if (!bias) return MOE_ERR_INVALID_ARG;
  return moe::permute_impl(xn, dtype, N, D, topk_idx, k, E, capacity, counts, offsets, row_map, perm_token, x_perm,
                           workspace, workspace_bytes, gamma, bias, max_over_mean_out, moe::as_cuda(stream));
}

extern "C" moe_status_t moe_permute(const void* xn, moe_dtype_t dtype, int N, int D,
                                    const int32_t* topk_idx, int k, int E, int32_t* counts,
                                    int32_t* offsets, int32_t* row_map, int32_t* perm_token,
                                    void* x_perm, void* workspace, size_t workspace_bytes,
                                    moe_stream_t stream) {
  return moe_permute_capacity(xn, dtype, N, D, topk_idx, k, E, 0x7fffffff, counts, offsets, row_map,
                              perm_token, x_perm, workspace, workspace_bytes, stream);
}

// ---- moe_permute_noalloc ---------------------------------------------------------------
// The same permutation for callers that cannot allocate device memory: its scratch lives
// in a fixed file-scope device array that every GPU loading the library holds until exit.
#include <mutex>

namespace moe {
namespace {

constexpr size_t kNoAllocScratchInts = 65536;  // 256 KiB
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

// Device address of g_permute_scratch on the current device, looked up once per device.
int32_t* noalloc_scratch() {
  static std::mutex mu;
  static int32_t* addr[128] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    int32_t* p = nullptr;
    if (cudaGetSymbolAddress((void**)&p, g_permute_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_permute_noalloc_max_scratch_bytes(void) {
  return moe::kNoAllocScratchInts * sizeof(int32_t);
}

extern "C" moe_status_t moe_permute_noalloc(const void* xn, moe_dtype_t dtype, int N, int D,
                                            const int32_t* topk_idx, int k, int E, int32_t* counts,
                                            int32_t* offsets, int32_t* row_map, int32_t* perm_token,
                                            void* x_perm, moe_stream_t stream) {
  using namespace moe;
  if (N < 0 || k < 1 || E < 1 || k > E || D <= 0) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_permute_workspace_bytes(N, k, E);
  if (need > kNoAllocScratchInts * sizeof(int32_t)) return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = noalloc_scratch();
  if (!scratch) return MOE_ERR_CUDA;
  return moe_permute(xn, dtype, N, D, topk_idx, k, E, counts, offsets, row_map, perm_token, x_perm,
                     scratch, kNoAllocScratchInts * sizeof(int32_t), stream);
}

// Router on tensor cores: fp32 router weights split exactly into three bf16 planes.
//
// Lesson "Mixture of Experts", "Build it" step 1 (router scores = dot products of the
// token with every expert's router row); handbook article, router-precision paragraph
// (bf16 rounding of close logits can change the winner, so the router must keep fp32
// accuracy).
//
// Every fp32 weight w is written as w = hi + mid + lo with three bf16 numbers (8
// significant bits each, exact for finite normal weights).  The activations are bf16,
// so every product x*hi, x*mid, x*lo is exact in fp32 and the tensor core computes
// sum_d x_d * (hi_d + mid_d + lo_d) with fp32 accumulation.  The tensor core's own
// accumulation over a long reduction is not correctly rounded (measured on B300: 7e-6 to
// 2e-5 rms logit error when one accumulator spans all of D), so:
//   * every 64-element slice of the reduction is summed in a fresh TMEM accumulator and
//     the epilogue warps add the slice partials in registers, with two-sum compensation
//     (measured 8e-8 rms for the hi plane alone, about the fp32 rounding of the result).
// The three planes sit one after another in shared memory, so one MMA with N = 3*NT
// covers all of them: 4 MMAs per slice.  The kernel is bound by issuing MMAs (one thread
// issues them, at a cost per instruction well above the execution time of a narrow MMA),
// which is why the planes share an instruction.  The hand-off per slice is one mbarrier
// arrival per epilogue warp and a plain add per column (hi + (mid + lo)), folded into the
// compensated total every 8 slices.  Short token counts are split along D (split-K) so that about
// 128 CTAs stream the activations; the top-k kernel adds the split partials in order.
//
// Kernels: split (w -> 3 bf16 planes), router GEMM (tcgen05, logits [N, E] fp32), and a
// warp-per-token top-k over the logits (shared selection code with the CUDA-core path).
#include <algorithm>

#include "tc_common.cuh"
#include "topk_common.cuh"

namespace moe {
namespace rtc {

using namespace moe::tc;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UK = 16;

__global__ void split_kernel(const float* __restrict__ w, long long n, __nv_bfloat16* __restrict__ out) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  grid_dep_wait();
  grid_dep_launch();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float x = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(hi);    // exact
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);  // exact, <= 8 significant bits
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

// NBUF slice accumulators in TMEM let the MMA warp run up to NBUF-1 slices ahead of the
// epilogue; EPI epilogue warps share the columns (two warps per TMEM lane quarter when 8).
// SH: the launch also runs the shared expert's first GEMM (below), whose stages hold a 256-row
// weight tile and whose accumulator takes 256 TMEM columns.
template <int NT, bool SH = false>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = NT * BK * 2;  // one split plane
  static constexpr int SH_B_BYTES = 256 * BK * 2;  // the shared expert's 128 gate + 128 up rows
  static constexpr int STAGE_BYTES = A_BYTES + (SH && SH_B_BYTES > 3 * B_BYTES ? SH_B_BYTES : 3 * B_BYTES);
  static constexpr int STAGES = NT >= 64 || SH ? 4 : 6;
  static constexpr int ACC = 3 * NT;                  // one slice accumulator: [hi | mid | lo]
  static constexpr int NBUF = 512 / ACC < 8 ? 512 / ACC : 8;  // slice accumulators in TMEM
  static constexpr int TMEM_COLS = SH ? 512 : (NBUF * ACC <= 256 ? (NBUF * ACC <= 128 ? 128 : 256) : 512);
  static constexpr int EPI = NT >= 32 ? 8 : 4;         // epilogue warps
  static constexpr int W = NT / (EPI / 4);             // columns per epilogue thread
  static constexpr int THREADS = 96 + 32 * EPI;       // + warp 2 + EPI: activation copies
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 512;
};

// The shared expert's part of a router launch (SH): its gate/up weights as a two-plane map with
// 128-row boxes, its d_ff, the plane order (1: gate first) and H = SiLU(x W_gate^T) * (x W_up^T)
// out, [N, F] bf16.
struct SharedUp {
  int et = 0;  // router expert tiles: grid.y beyond them are the shared expert's column blocks
  int F = 0;
  int planes = 0;
  __nv_bfloat16* h = nullptr;
};

// Start loading 16 consecutive fp32 TMEM columns of this warp's lane quarter (complete
// with tmem_ld_wait()).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// One 128-token x 128-output tile of the shared expert's first GEMM inside a router launch:
// warp 0 copies the gate/up rows (one two-plane box per 64-wide k-block), the last warp the
// tokens, warp 1 issues M = 128, N = 256 MMAs into TMEM columns [0, 256) over all of D, and
// the epilogue warps apply SwiGLU and store H in bf16 (rows past N and outputs past F are
// not written).  Uses the launch's stage ring and barriers from their initial phase.
template <class C>
__device__ __forceinline__ void shared_up_tile(uint8_t* smem, uint64_t* bars, uint32_t tmem_base,
                                               volatile int* abort_flag, const CUtensorMap& map_x,
                                               const CUtensorMap& map_s, const SharedUp& sh, int N, int D, int m0,
                                               int* status) {
  constexpr int STAGES = C::STAGES;
  constexpr uint32_t IDESC_SH = idesc_bf16(BM, 256);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  constexpr int A_WARP = 2 + C::EPI;
  const int n0 = ((int)blockIdx.y - sh.et) * 128;  // first output (gate / up row) of this tile
  const int KB = D / BK;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  const uint32_t tfull = smem_u32(bars + 2 * STAGES);  // the first slice barrier serves the tile
  const uint32_t done_bar = smem_u32(bars + 2 * STAGES + 2 * C::NBUF);
  if ((warp == 0 || warp == A_WARP) && lane == 0) {
    const bool is_w = warp == 0;
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    for (int kb = 0; kb < KB; ++kb) {
      if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status, true)) break;
      const uint32_t a_dst = smem_u32(smem + stage * C::STAGE_BYTES);
      if (is_w) {
        mbar_expect_tx(full_bar(stage), C::SH_B_BYTES);
        tma_load_3d(a_dst + C::A_BYTES, &map_s, kb * BK, n0, 0, full_bar(stage));
      } else {
        mbar_expect_tx(full_bar(stage), C::A_BYTES);
        tma_load_2d(a_dst, &map_x, kb * BK, m0, full_bar(stage));
      }
      issued |= 1u << stage;
      issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) { stage = 0; phase ^= 1u; }
    }
    for (int s = 0; s < STAGES; ++s)
      if ((issued >> s) & 1u) mbar_wait(full_bar(s), (issued_par >> s) & 1u, abort_flag, status, false);
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < KB && ok; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag, status, true)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
        const uint32_t b_base = a_base + C::A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UK; ++k)
          tc_mma(tmem_base, sw128_desc(a_base + k * UK * 2), sw128_desc(b_base + k * UK * 2), IDESC_SH,
                 (kb | k) != 0 ? 1u : 0u);
        tc_commit(empty_bar(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (ok) tc_commit(tfull);
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, abort_flag, status, false);
    }
  } else if (warp >= 2 && warp < A_WARP) {
    constexpr int PER_Q = C::EPI / 4;       // epilogue warps per TMEM lane quarter
    constexpr int OUTS = 128 / PER_Q;       // outputs per warp
    const int q = warp & 3, part = (warp - 2) >> 2;
    const int row = m0 + q * 32 + lane;
    const uint32_t gcol = sh.planes == 2 ? 128u : 0u;  // up rows came first in B when 2
    int got = 1;
    if (lane == 0) got = mbar_wait(tfull, 0, abort_flag, status, true) ? 1 : 0;
    __syncwarp();
    if (__shfl_sync(0xffffffffu, got, 0) != 0) {
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c0 = part * OUTS; c0 < (part + 1) * OUTS; c0 += 32) {
        uint32_t gv[32], uv[32];
        tmem_ld32(taddr + gcol + (uint32_t)c0, gv);
        tmem_ld32(taddr + (128u - gcol) + (uint32_t)c0, uv);
        tmem_ld_wait();
        uint4 packed[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float hv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float g = __uint_as_float(gv[v * 8 + i]);
            const float uu = __uint_as_float(uv[v * 8 + i]);
            hv[i] = __fdividef(g, 1.0f + __expf(-g)) * uu;
          }
          packed[v] = f32_to_bf16x8(hv);
        }
        if (row < N && n0 + c0 < sh.F) {  // F is a multiple of 64, so a 32-output chunk is whole
          uint4* dst = reinterpret_cast<uint4*>(sh.h + (size_t)row * sh.F + n0 + c0);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = packed[v];
        }
      }
    }
  }
}

// grid (ceil(N/128), ceil(E/NT) [+ ceil(F/128) with SH], splits); block = TMA warp, MMA warp,
// EPI epilogue warps.
//
// SH (router rows and the shared expert's gate/up rows in one launch; handbook news article,
// the fused-permute paragraph: bytes moved around the expert GEMMs cost): a CTA with
// blockIdx.y >= sh.et computes the shared expert's first GEMM for its 128 tokens and 128
// outputs (blockIdx.y - sh.et), H = SiLU(acc[:, gate]) * acc[:, up] over all of D in one
// 256-column accumulator, with the same MMA sequence and epilogue arithmetic as the grouped
// SwiGLU kernel (the same bits).  Its token tiles are the router's: every token block's rows
// come from HBM once and from L2 for the other CTAs of that block.
template <int NT, bool SH = false>
__global__ void __launch_bounds__(Cfg<NT, SH>::THREADS, 1)
router_gemm_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                   int N, int D, int E, int kb_per_split,
                   float* __restrict__ logits, float* __restrict__ partials, int* __restrict__ status,
                   const __grid_constant__ CUtensorMap map_s, SharedUp sh) {
  using C = Cfg<NT, SH>;
  constexpr uint32_t IDESC = idesc_bf16(BM, 3 * NT);
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int NBUF = C::NBUF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[NBUF], tempty[NBUF], done
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2 * NBUF + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int m0 = blockIdx.x * BM, e0 = blockIdx.y * NT;
  const int kb0 = blockIdx.z * kb_per_split;
  const int kb1 = min(D / BK, kb0 + kb_per_split);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + NBUF + a); };
  const uint32_t done_bar = smem_u32(bars + 2 * STAGES + 2 * NBUF);

  if (t == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 2);  // weight-plane copies (warp 0) + activation copies (last warp)
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < NBUF; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), C::EPI);  // one arrival per epilogue warp
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  grid_dep_wait();  // barriers and tensor memory are set up; from here on the inputs are read
  grid_dep_launch();

  constexpr int A_WARP = 2 + C::EPI;
  if constexpr (SH) {
    if ((int)blockIdx.y >= sh.et) {
      if (blockIdx.z == 0) shared_up_tile<C>(smem, bars, tmem_base, abort_flag, map_x, map_s, sh, N, D, m0, status);
      tc_fence_before();
      __syncthreads();
      if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::TMEM_COLS));
      }
      return;
    }
  }
  if ((warp == 0 || warp == A_WARP) && lane == 0) {
    // warp 0: the three weight planes of the slice as one 3-D box; last warp: the tokens
    const bool is_w = warp == 0;
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    {
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status, true)) break;
        const uint32_t a_dst = smem_u32(smem + stage * C::STAGE_BYTES);
        if (is_w) {
          mbar_expect_tx(full_bar(stage), 3 * C::B_BYTES);
          tma_load_3d(a_dst + C::A_BYTES, &map_w, kb * BK, e0, 0, full_bar(stage));
        } else {
          mbar_expect_tx(full_bar(stage), C::A_BYTES);
          tma_load_2d(a_dst, &map_x, kb * BK, m0, full_bar(stage));
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(full_bar(s), (issued_par >> s) & 1u, abort_flag, status, false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, status, true)) break;
        if (!mbar_wait(full_bar(stage), phase, abort_flag, status, true)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
        const uint32_t b_base = a_base + C::A_BYTES;  // [hi ; mid ; lo], NT rows each
#pragma unroll
        for (int k = 0; k < BK / UK; ++k) {
          const uint64_t ad = sw128_desc(a_base + k * UK * 2);
          tc_mma(tmem_base + (uint32_t)(acc * C::ACC), ad, sw128_desc(b_base + k * UK * 2), IDESC, k ? 1u : 0u);
        }
        tc_commit(empty_bar(stage));
        tc_commit(tfull_bar(acc));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        if (++acc == NBUF) { acc = 0; acc_phase ^= 1u; }
      }
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, abort_flag, status, false);
    }
  } else if (warp >= 2 && warp < A_WARP) {
    constexpr int W = C::W;
    const int q = warp & 3;                // TMEM lane quarter
    const int cb = ((warp - 2) >> 2) * W;  // this warp's first column
    const int row = m0 + q * 32 + lane;
    // Slice partials are added plainly into `loc` (8 slices at most), and every 8 slices
    // `loc` is folded into the running total with a two-sum (s, c).
    float s[W], c[W], loc[W];
#pragma unroll
    for (int j = 0; j < W; ++j) s[j] = c[j] = loc[j] = 0.f;
    auto fold = [&]() {
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const float a = s[j], b = loc[j];
        const float tt = a + b;
        const float bp = tt - a;
        c[j] += (a - (tt - bp)) + (b - bp);
        s[j] = tt;
        loc[j] = 0.f;
      }
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb) {
      // lane 0 watches the barrier; the warp follows through __syncwarp
      int got = 1;
      if (lane == 0) got = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, status, true) ? 1 : 0;
      __syncwarp();
      ok = __shfl_sync(0xffffffffu, got, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      // this slice's partials of the three planes, 16 columns at a time: hi + (mid + lo)
      const uint32_t ab = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::ACC + cb);
#pragma unroll
      for (int h = 0; h < W; h += 16) {
        uint32_t rh[16], rm[16], rl[16];
        tmem_ld16(ab + (uint32_t)h, rh);
        tmem_ld16(ab + (uint32_t)(NT + h), rm);
        tmem_ld16(ab + (uint32_t)(2 * NT + h), rl);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          loc[h + j] += __uint_as_float(rh[j]) + (__uint_as_float(rm[j]) + __uint_as_float(rl[j]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (((kb - kb0) & 7) == 7) fold();
      if (++acc == NBUF) { acc = 0; acc_phase ^= 1u; }
    }
    fold();
    if (ok && row < N) {
      const int e1 = e0 + cb;
      float* dst = (blockIdx.z == 0 ? logits : partials + (size_t)(blockIdx.z - 1) * N * E) + (size_t)row * E + e1;
      if (e1 + W <= E && (E & 3) == 0) {
#pragma unroll
        for (int j = 0; j < W; j += 4)
          *reinterpret_cast<float4*>(dst + j) =
              make_float4(s[j] + c[j], s[j + 1] + c[j + 1], s[j + 2] + c[j + 2], s[j + 3] + c[j + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < W; ++j)
          if (e1 + j < E) dst[j] = s[j] + c[j];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::TMEM_COLS));
  }
}

// warp per token over the logits
template <int PER>
__global__ void __launch_bounds__(256) topk_kernel(float* __restrict__ logits, const float* __restrict__ partials,
                                                   int nsplit, const float* __restrict__ bias, int N, int E, int k,
                                                   int score_fn, int32_t* __restrict__ idx, float* __restrict__ gate,
                                                   uint8_t* __restrict__ tie, int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  grid_dep_wait();
  grid_dep_launch();
  if (n >= N) return;
  float* row = logits + (size_t)n * E;
  float lg[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? row[e] : 0.f;
  }
  if (nsplit > 1) {  // add the split-K partials in split order (two-sum), write the logits
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (e >= E) continue;
      float sum = lg[i], comp = 0.f;
      for (int z = 1; z < nsplit; ++z) {
        const float b = partials[((size_t)(z - 1) * N + n) * E + e];
        const float tt = sum + b;
        const float bp = tt - sum;
        comp += (sum - (tt - bp)) + (b - bp);
        sum = tt;
      }
      lg[i] = sum + comp;
      row[e] = lg[i];
    }
  }
  warp_topk_gates<PER>(lg, lane, E, k, bias, score_fn, idx + (size_t)n * k, gate + (size_t)n * k,
                       tie ? tie + n : nullptr, status);
}

// With SH, grid.y also covers the shared expert's ceil(F / 128) output blocks after the
// router's expert tiles (`ms` its gate/up map, `sh` its sizes and output).
template <int NT, bool SH = false>
moe_status_t launch_gemm(const CUtensorMap& mx, const CUtensorMap& mw, int N, int D, int E, int nsplit,
                         float* logits, float* partials, int* status, cudaStream_t s, const CUtensorMap& ms,
                         SharedUp sh) {
  using C = Cfg<NT, SH>;
  auto kern = router_gemm_kernel<NT, SH>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int KB = D / BK;
  const int per = (KB + nsplit - 1) / nsplit;
  sh.et = (E + NT - 1) / NT;
  dim3 grid((N + BM - 1) / BM, sh.et + (SH ? (sh.F + 127) / 128 : 0), nsplit);
  return launch_kernel(kern, grid, dim3(C::THREADS), C::SMEM, s, mx, mw, N, D, E, per, logits, partials, status, ms,
                       sh);
}

// Tile width and split-K count for (N, D, E): about 128 CTAs, at most 4 splits.
struct Plan {
  int nt, nsplit;
};

Plan plan(int N, int D, int E) {
  Plan p;
  const int mt = (N + BM - 1) / BM;
  p.nt = E <= 16 ? 16 : (E <= 32 ? 32 : 64);
  const int ctas = mt * ((E + p.nt - 1) / p.nt);
  const int KB = D / BK;
  p.nsplit = std::max(1, std::min(std::min(4, KB), (128 + ctas - 1) / ctas));
  // every split must own at least one k-block
  while (p.nsplit > 1 && (KB + p.nsplit - 1) / p.nsplit * (p.nsplit - 1) >= KB) --p.nsplit;
  return p;
}

}  // namespace rtc
}  // namespace moe

extern "C" size_t moe_router_split_bytes(int E, int D) {
  if (E <= 0 || D <= 0) return 0;
  return (size_t)3 * E * D * sizeof(uint16_t);
}

extern "C" moe_status_t moe_router_split(const float* w_router, int E, int D, void* w_split,
                                         moe_stream_t stream) {
  using namespace moe;
  if (E < 1 || D < 1 || !w_router || !w_split) return MOE_ERR_INVALID_ARG;
  const long long n = (long long)E * D;
  const int blocks = (int)std::min<long long>((n + 255) / 256, (long long)sm_count() * 8);
  return launch_kernel(rtc::split_kernel, dim3(blocks), dim3(256), 0, as_cuda(stream), w_router, n,
                       static_cast<__nv_bfloat16*>(w_split));
}

extern "C" size_t moe_router_topk_split_workspace_bytes(int N, int D, int E) {
  if (N <= 0 || D <= 0 || E <= 0 || D % 64 != 0) return 0;
  const moe::rtc::Plan p = moe::rtc::plan(N, D, E);
  return (size_t)(p.nsplit - 1) * N * E * sizeof(float);
}

namespace moe {
namespace rtc {
namespace {
// moe_router_topk_split, and with ws_gate the shared expert's first GEMM in the same launch.
moe_status_t router_impl(const void* xn, int N, int D, const void* w_split, const float* bias, int E, int k,
                         moe_score_fn_t fn, float* logits_out, int32_t* topk_idx, float* topk_gate,
                         uint8_t* near_tie, void* workspace, size_t workspace_bytes, const void* ws_gate,
                         const void* ws_up, int F, void* hs_out, moe_stream_t stream) {
  const bool with_shared = ws_gate != nullptr;
  if (N < 0 || D <= 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > MOE_MAX_EXPERTS || k > MOE_MAX_TOPK || D % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (fn != MOE_SCORE_SOFTMAX && fn != MOE_SCORE_SIGMOID && fn != MOE_SCORE_SQRT_SOFTPLUS) return MOE_ERR_INVALID_ARG;
  if (with_shared && (F <= 0 || !ws_up || !hs_out)) return MOE_ERR_INVALID_ARG;
  if (with_shared && F % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (!xn || !w_split || !logits_out || !topk_idx || !topk_gate) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xn) || !aligned16(w_split) || !aligned16(logits_out)) return MOE_ERR_INVALID_ARG;
  if (with_shared && (!aligned16(ws_gate) || !aligned16(ws_up) || !aligned16(hs_out))) return MOE_ERR_INVALID_ARG;
  const Plan p = plan(N, D, E);
  if (p.nsplit > 1 && (!workspace || workspace_bytes < moe_router_topk_split_workspace_bytes(N, D, E)))
    return MOE_ERR_INVALID_ARG;
  int* status = device_status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = as_cuda(stream);
  CUtensorMap mx, mw, ms;
  if (!tc::make_map_bf16(&mx, xn, (uint64_t)N, (uint64_t)D, BM) ||
      !tc::make_map_planes_bf16(&mw, w_split, (uint64_t)E, (uint64_t)D, 3, (uint32_t)p.nt))
    return MOE_ERR_CUDA;
  SharedUp sh;
  if (with_shared) {
    if (!tc::make_map_gate_up(&ms, ws_gate, ws_up, (uint64_t)F, (uint64_t)D, 128, &sh.planes))
      return MOE_ERR_UNSUPPORTED;  // the shared gate/up pair must form one two-plane map
    sh.F = F;
    sh.h = static_cast<__nv_bfloat16*>(hs_out);
  } else {
    ms = mx;  // not read
  }
  float* part = static_cast<float*>(workspace);
  moe_status_t st;
  if (with_shared)
    st = p.nt == 16 ? launch_gemm<16, true>(mx, mw, N, D, E, p.nsplit, logits_out, part, status, s, ms, sh)
         : p.nt == 32 ? launch_gemm<32, true>(mx, mw, N, D, E, p.nsplit, logits_out, part, status, s, ms, sh)
                      : launch_gemm<64, true>(mx, mw, N, D, E, p.nsplit, logits_out, part, status, s, ms, sh);
  else
    st = p.nt == 16 ? launch_gemm<16>(mx, mw, N, D, E, p.nsplit, logits_out, part, status, s, ms, sh)
         : p.nt == 32 ? launch_gemm<32>(mx, mw, N, D, E, p.nsplit, logits_out, part, status, s, ms, sh)
                      : launch_gemm<64>(mx, mw, N, D, E, p.nsplit, logits_out, part, status, s, ms, sh);
  if (st != MOE_OK) return st;
  const int sig = (int)fn;  // score function code
  const int grid = (N + 7) / 8;
  auto topk = [&](auto kern) {
    return launch_kernel(kern, dim3(grid), dim3(256), 0, s, logits_out, static_cast<const float*>(part), p.nsplit,
                         bias, N, E, k, sig, topk_idx, topk_gate, near_tie, status);
  };
  if (E <= 32) return topk(topk_kernel<1>);
  if (E <= 64) return topk(topk_kernel<2>);
  if (E <= 128) return topk(topk_kernel<4>);
  if (E <= 256) return topk(topk_kernel<8>);
  if (E <= 512) return topk(topk_kernel<16>);
  return topk(topk_kernel<32>);
}
}  // namespace
}  // namespace rtc
}  // namespace moe

extern "C" moe_status_t moe_router_topk_split(const void* xn, int N, int D, const void* w_split,
                                              const float* bias, int E, int k, moe_score_fn_t fn,
                                              float* logits_out, int32_t* topk_idx, float* topk_gate,
                                              uint8_t* near_tie, void* workspace, size_t workspace_bytes,
                                              moe_stream_t stream) {
  return moe::rtc::router_impl(xn, N, D, w_split, bias, E, k, fn, logits_out, topk_idx, topk_gate, near_tie,
                               workspace, workspace_bytes, nullptr, nullptr, 0, nullptr, stream);
}

extern "C" moe_status_t moe_router_topk_split_shared(const void* xn, int N, int D, const void* w_split,
                                                     const float* bias, int E, int k, moe_score_fn_t fn,
                                                     float* logits_out, int32_t* topk_idx, float* topk_gate,
                                                     uint8_t* near_tie, void* workspace, size_t workspace_bytes,
                                                     const void* ws_gate, const void* ws_up, int F, void* hs_out,
                                                     moe_stream_t stream) {
  if (!ws_gate) return MOE_ERR_INVALID_ARG;
  return moe::rtc::router_impl(xn, N, D, w_split, bias, E, k, fn, logits_out, topk_idx, topk_gate, near_tie,
                               workspace, workspace_bytes, ws_gate, ws_up, F, hs_out, stream);
}

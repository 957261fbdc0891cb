// Grouped SwiGLU expert FFN over ragged per-expert row blocks.
//
// Lesson "Mixture of Experts", section "Concept": every expert is an independent
// SwiGLU FFN, y = W_down (SiLU(W_gate x) * (W_up x)); section "Shared experts": the
// always-on expert is the same computation with one group covering every token.
//
// bf16 path: two launches of one persistent, warp-specialised tcgen05 kernel.
//   GEMM1  acc[128 x 256] = X[rows] . [W_gate[n0:n0+128] ; W_up[n0:n0+128]]^T
//          epilogue H = SiLU(acc[:, :128]) * acc[:, 128:]  -> bf16
//   GEMM2  acc[128 x 256] = H[rows] . W_down[n0:n0+256]^T  -> bf16 Y
// Roles (192 threads, one CTA per SM):
//   warp 0      one lane issues TMA loads (128B-swizzled K-major tiles) into a
//               4-stage shared-memory ring guarded by full/empty mbarriers;
//   warp 1      allocates 512 TMEM columns (two 256-column fp32 accumulators) and
//               one lane issues tcgen05.mma (M=128, or M=64 for a tile of at most 64
//               rows; N=256, K=16) and tcgen05.commit;
//   warps 2..5  drain an accumulator with tcgen05.ld while the MMA warp fills the
//               other one, apply the epilogue and store bf16 rows, masking rows past
//               the expert's segment and columns past the output width.
// Tiles are (expert g, column block, 128-row block) with the row block fastest, so
// CTAs running at the same time share weight tiles through L2.  The tile list comes
// from the device-side offsets: every CTA scans them into shared memory at start.
// Every mbarrier wait is bounded in wall time; on expiry the kernel records
// MOE_ERR_TIMEOUT in the status word, lets in-flight copies and MMAs land, frees
// its TMEM and returns.
//
// fp32 path: tiled CUDA-core kernels (64 x 64 output tiles, fp32 FMA chains in K order).
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tc_common.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;                 // rows per tile (UMMA M)
constexpr int BN = 256;                 // accumulator columns (UMMA N)
constexpr int BK = 64;                  // K per stage: one 128-byte swizzle row of bf16
constexpr int UK = 16;                  // K per tcgen05.mma (bf16)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int B_BYTES = BN * BK * 2;    // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int MAX_GROUPS = 1024;
constexpr int STAGING_BYTES = 32 * 128;  // one 32-row x 64-column bf16 output block

constexpr uint32_t IDESC = idesc_bf16(BM, BN);
// A tile with at most 64 rows (an expert's last rows, a small expert) is a half tile: one
// M = 64 MMA per K step instead of an M = 128 one over 64 or more padded rows.  Measured on
// B300 (N = 256, K = 16) it takes the same 128 cycles as M = 128 but draws less power, which
// is what sets the speed of these launches once the GPU runs at its power limit.  (The
// weight-stationary M = 64 form takes 80 cycles but drew more power: slower at the limit.)
// Measured accumulator layout (M = 64, one CTA): row r sits in TMEM lane 32 * (r / 16) +
// r % 16, at the same columns as for M = 128.
constexpr int HALF_ROWS = BM / 2;
constexpr uint32_t IDESC_HALF = idesc_bf16(HALF_ROWS, BN);
constexpr int A_BOX = HALF_ROWS;        // rows per A copy: one for a half tile, two for a full one

// Most CTAs a grouped GEMM launch may use (0 = every SM); set for one call by
// moe_grouped_swiglu_ex so that other work can run on the remaining SMs.
thread_local int g_max_ctas = 0;
inline int cta_cap() { return g_max_ctas > 0 ? std::min(g_max_ctas, sm_count()) : sm_count(); }

struct Tile {
  int g, row0, rows, nb, mb;
  int x;  // 1: a tile of the extra group (the shared expert run in the same launch)
};

template <int ROWS>
__device__ __forceinline__ Tile decode_rows(int tile, const int* tile_start, int G, const int32_t* offsets,
                                            int M_total, int NB) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  Tile t;
  t.g = lo;
  t.x = 0;
  const int s = min(max(__ldg(offsets + lo), 0), M_total);
  const int e = min(max(__ldg(offsets + lo + 1), s), M_total);
  const int mblk = (e - s + ROWS - 1) / ROWS;
  const int local = tile - tile_start[lo];
  t.nb = local / mblk;
  const int mb = local - t.nb * mblk;
  t.mb = mb;
  t.row0 = s + mb * ROWS;
  t.rows = min(ROWS, e - t.row0);
  return t;
}

__device__ __forceinline__ Tile decode(int tile, const int* tile_start, int G, const int32_t* offsets,
                                       int M_total, int NB) {
  return decode_rows<BM>(tile, tile_start, G, offsets, M_total, NB);
}

// The tile list of a launch that also runs an extra group (the shared expert: rows [0, M2) of
// its own operands): the `routed` tiles of the groups, then NX = ceil(M2/128) * NB extra tiles,
// which fill the routed tiles' last wave.  (Spreading the extra tiles evenly among the routed
// ones, with the routed weights marked evict-first and the shared operands evict-last in L2,
// measured 16 % slower on the DeepSeek-V3 layer: the streamed weights still pushed the shared
// operands out of L2.)
struct ExtraList {
  int routed, NX, M2;
  __device__ __forceinline__ int total() const { return routed + NX; }
};

__device__ __forceinline__ Tile decode_list(int t, const ExtraList& L, const int* tile_start, int G,
                                            const int32_t* offsets, int M_total, int NB) {
  if (t < L.routed) return decode(t, tile_start, G, offsets, M_total, NB);
  const int xi = t - L.routed;
  Tile r;
  const int mblk = (L.M2 + BM - 1) / BM;
  r.g = 0;
  r.x = 1;
  r.nb = xi / mblk;
  r.mb = xi - r.nb * mblk;
  r.row0 = r.mb * BM;
  r.rows = min(BM, L.M2 - r.row0);
  return r;
}

// MODE 0: GEMM1 with SwiGLU epilogue (B = gate rows ; up rows, 128 output columns per tile)
// MODE 1: GEMM2 (B = 256 rows of W_down, 256 output columns per tile)
// MODE 2: MODE 0 with the A rows gathered from xn through perm_token (no permuted copy).
//         Warps 6..9 copy 32 tile rows each with 16-byte cp.async into the 128-byte-swizzled
//         K-major layout the MMA descriptors expect; each thread keeps LAG k-blocks of copies
//         in flight, then waits for the oldest, fences the async proxy and arrives on that
//         stage's full barrier (initialised for 1 + 128 arrivals).
//         LAG <= STAGES - 2 keeps one k-block queued on the tensor pipe while a stage fills:
//         the arrival for stage s needs the MMA of stage s + LAG - STAGES to have completed.
// Warp 6 (MODE 0/1) issues the A-tile copies while warp 0 issues the B-tile copies: one
// thread issuing every copy of a stage leaves the copy engine underused (measured).
template <int MODE>
constexpr int kThreads = MODE == 2 ? THREADS + 128 : THREADS + 32;
#ifndef MOE_GATHER_LAG
#define MOE_GATHER_LAG (STAGES - 2)
#endif
constexpr int GATHER_LAG = MOE_GATHER_LAG;
static_assert(GATHER_LAG >= 0 && GATHER_LAG < STAGES, "gather lag must leave a stage to wait on");

template <int MODE>
__global__ void __launch_bounds__(kThreads<MODE>, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                    const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_out,
                    const int32_t* __restrict__ offsets, int G, int M_total, int K, int NOUT,
                    __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ xg, int NX,
                    const int32_t* __restrict__ perm, int b_planes, int nbuf, int* __restrict__ status,
                    const __grid_constant__ CUtensorMap map_a2, const __grid_constant__ CUtensorMap map_b2,
                    const __grid_constant__ CUtensorMap map_out2, int M2, __nv_bfloat16* __restrict__ out2,
                    int b2_planes) {
  constexpr bool SWIGLU = MODE != 1;
  constexpr int TN = SWIGLU ? BN / 2 : BN;  // output columns per tile
  constexpr int NTHR = kThreads<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // output staging: nbuf 4 KB buffers (32 rows x 64 bf16, 128-byte swizzle) per epilogue warp
  uint8_t* staging = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + 4 * nbuf * STAGING_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], done
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* wtot = reinterpret_cast<int*>(tmem_holder + 2);  // [16]
  int* tile_start = wtot + 16;                           // [G + 1]

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int NB = (NOUT + TN - 1) / TN;
  const int KB = K / BK;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 2 + a); };
  const uint32_t done_bar = smem_u32(bars + 2 * STAGES + 4);

  if (t == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), MODE == 2 ? 1 + 128 : 2);  // B copies + A copies (or one per gather thread)
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);  // one arrival per epilogue warp
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == 6 && lane == 0 && MODE != 2)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b0)) : "memory");
    if (SWIGLU) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b1)) : "memory");
  }

  grid_dep_wait();  // set-up done; the offsets and operands come from earlier kernels
  grid_dep_launch();

  // tile_start[g] = sum over g' < g of (row blocks of g') * NB
  {
    const int per = (G + NTHR - 1) / NTHR;
    const int g0 = min(G, t * per), g1 = min(G, g0 + per);
    int local = 0;
    for (int g = g0; g < g1; ++g) {
      const int s = min(max(__ldg(offsets + g), 0), M_total);
      const int e = min(max(__ldg(offsets + g + 1), s), M_total);
      local += ((e - s + BM - 1) / BM) * NB;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += wtot[w];
    base += incl - local;
    for (int g = g0; g < g1; ++g) {
      tile_start[g] = base;
      const int s = min(max(__ldg(offsets + g), 0), M_total);
      const int e = min(max(__ldg(offsets + g + 1), s), M_total);
      base += ((e - s + BM - 1) / BM) * NB;
    }
    if (t == NTHR - 1) {
      int tot = 0;
      for (int w = 0; w < NTHR / 32; ++w) tot += wtot[w];
      tile_start[G] = tot;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  ExtraList XL;
  XL.routed = tile_start[G];
  XL.M2 = M2;
  XL.NX = XL.M2 > 0 ? ((XL.M2 + BM - 1) / BM) * NB : 0;
  const int total_tiles = XL.total();
  auto tile_at = [&](int tile) { return decode_list(tile, XL, tile_start, G, offsets, M_total, NB); };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: weight (B) tiles ----------------
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const Tile tl = tile_at(tile);
        const int brow = (tl.x ? 0 : tl.g * NOUT) + tl.nb * TN;
        const CUtensorMap* mb = tl.x ? &map_b2 : &map_b0;
        const int planes = tl.x ? b2_planes : b_planes;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status, true)) { ok = false; break; }
          const uint32_t a_dst = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_dst = a_dst + A_BYTES;
          mbar_expect_tx(full_bar(stage), B_BYTES);
          if (SWIGLU && planes != 0) {  // gate and up rows as the two planes of one box
            tma_load_3d(b_dst, mb, kb * BK, brow, 0, full_bar(stage));
          } else if (SWIGLU) {
            tma_load_2d(b_dst, &map_b0, kb * BK, brow, full_bar(stage));
            tma_load_2d(b_dst + B_BYTES / 2, &map_b1, kb * BK, brow, full_bar(stage));
          } else {
            tma_load_2d(b_dst, mb, kb * BK, brow, full_bar(stage));
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // let every issued copy land before the CTA can exit
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(full_bar(s), (issued_par >> s) & 1u, abort_flag, status, false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const uint32_t idesc = tile_at(tile).rows <= HALF_ROWS ? IDESC_HALF : IDESC;
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, status, true)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, status, true)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UK; ++k)
            tc_mma(d_tmem, sw128_desc(a_base + k * UK * 2), sw128_desc(b_base + k * UK * 2), idesc,
                   (kb | k) != 0 ? 1u : 0u);
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      // every MMA issued so far completes before TMEM is freed
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, abort_flag, status, false);
    }
  } else if (MODE != 2 && warp == 6) {
    if (lane == 0) {
      // ---------------- TMA producer: activation (A) tiles ----------------
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const Tile tl = tile_at(tile);
        const CUtensorMap* ma = tl.x ? &map_a2 : &map_a;
        const bool half = tl.rows <= HALF_ROWS;  // the M = 64 MMA reads the first 64 rows only
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status, true)) { ok = false; break; }
          const uint32_t dst = smem_u32(smem + stage * STAGE_BYTES);
          mbar_expect_tx(full_bar(stage), half ? A_BYTES / 2 : A_BYTES);
          tma_load_2d(dst, ma, kb * BK, tl.row0, full_bar(stage));
          if (!half) tma_load_2d(dst + A_BYTES / 2, ma, kb * BK, tl.row0 + A_BOX, full_bar(stage));
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(full_bar(s), (issued_par >> s) & 1u, abort_flag, status, false);
    }
  } else if (MODE == 2 && warp >= 6) {
    // ---------------- A gather (warps 6..9): 32 tile rows per warp ----------------
    // Copy i of a lane moves 16 bytes (chunk lane % 8) of tile row 32 * w + 4 * i + lane / 8,
    // so each warp-wide copy reads four whole 128-byte row segments.
    constexpr int LAG = GATHER_LAG;
    const int w = warp - 6, c = lane & 7;
    int stage = 0, pend = 0, oldest = 0;
    uint32_t phase = 0;
    bool ok = true;
    // The next tile is decoded, and its token indices loaded, one tile ahead (in two steps,
    // after this tile's second and third k-blocks) so that a thread never stalls on those
    // dependent loads while earlier stages still wait for its arrival.
    Tile tl_next{};
    int tok_next[8];
    auto load_tokens = [&]() {  // the extra group's rows are xn's own rows, in order
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 32 * w + 4 * i + (lane >> 3);
        tok_next[i] = r < tl_next.rows ? (tl_next.x ? tl_next.row0 + r : __ldg(perm + tl_next.row0 + r)) : -1;
      }
    };
    const int kb_decode = KB > 2 ? 1 : 0, kb_tokens = KB > 2 ? 2 : KB - 1;
    if (blockIdx.x < total_tiles) {
      tl_next = tile_at(blockIdx.x);
      load_tokens();
    }
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
      const Tile tl = tl_next;
      const __nv_bfloat16* src[8];
      uint32_t live = 0, doff[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 32 * w + 4 * i + (lane >> 3);
        int tok = tok_next[i];
        if (r < tl.rows && (unsigned)tok >= (unsigned)NX) {  // not a token of xn: zero row, flagged
          if (c == 0) atomicOr(status, kStatusBadToken);
          tok = -1;
        }
        src[i] = xg + (size_t)(tok < 0 ? 0 : tok) * K + c * 8;
        live |= (tok < 0 ? 0u : 1u) << i;  // rows past the group are zero-filled, not read
        doff[i] = (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
      }
      const bool more = tile + (int)gridDim.x < total_tiles;
      const bool idle = tl.rows <= HALF_ROWS && w >= 2;  // rows 64..127: not read by the M = 64 MMA
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status, true)) { ok = false; break; }
        const uint32_t base = smem_u32(smem + stage * STAGE_BYTES);
        if (!idle) {
#pragma unroll
          for (int i = 0; i < 8; ++i) cp_async_16(base + doff[i], src[i] + kb * BK, ((live >> i) & 1u) << 4);
        }
        cp_async_commit();
        if (++pend > LAG) {  // the oldest stage's copies are complete once LAG groups remain
          cp_async_wait<LAG>();
          fence_proxy_async_smem();
          mbar_arrive(full_bar(oldest));
          if (++oldest == STAGES) oldest = 0;
          --pend;
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        if (more) {
          if (kb == kb_decode) tl_next = tile_at(tile + gridDim.x);
          if (kb == kb_tokens) load_tokens();
        }
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (; pend > 0; --pend) {
      mbar_arrive(full_bar(oldest));
      if (++oldest == STAGES) oldest = 0;
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    // Each warp owns 32 rows of the tile and writes them in 64-column blocks through a
    // swizzled shared-memory buffer and one TMA bulk store (row by row from registers when
    // the block crosses the end of its group's rows), as in the CTA-pair kernel.
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t my_staging = smem_u32(staging) + (uint32_t)(q * nbuf * STAGING_BYTES);
    int acc = 0, bi = 0, stores = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const Tile tl = tile_at(tile);
      const uint32_t gcol = (tl.x ? b2_planes : b_planes) == 2 ? TN : 0;  // up rows came first in B
      const CUtensorMap* mo = tl.x ? &map_out2 : &map_out;
      __nv_bfloat16* optr = tl.x ? out2 : out;
      const bool ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, status, true);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      // a half tile's rows 16q..16q+15 are in this warp's lanes 0..15
      const bool half = tl.rows <= HALF_ROWS;
      const int r0 = half ? q * 16 : q * 32;  // first tile row of this warp
      const bool valid = (!half || lane < 16) && r0 + lane < tl.rows;
      const bool whole = !half && r0 + 32 <= tl.rows;  // warp-uniform
#pragma unroll 1
      for (int u = 0; u < TN / 64; ++u) {
        const int ocol = u * 64;
        if (tl.nb * TN + ocol >= NOUT) continue;  // column tail (warp-uniform)
        uint4 packed[8];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (SWIGLU) {
            uint32_t gv[32], uv[32];
            tmem_ld32(taddr + gcol + ocol + c * 32, gv);
            tmem_ld32(taddr + (TN - gcol) + ocol + c * 32, uv);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float h[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float g = __uint_as_float(gv[v * 8 + i]);
                const float uu = __uint_as_float(uv[v * 8 + i]);
                h[i] = __fdividef(g, 1.0f + __expf(-g)) * uu;
              }
              packed[c * 4 + v] = f32_to_bf16x8(h);
            }
          } else {
            uint32_t yv[32];
            tmem_ld32(taddr + ocol + c * 32, yv);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float y[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) y[i] = __uint_as_float(yv[v * 8 + i]);
              packed[c * 4 + v] = f32_to_bf16x8(y);
            }
          }
        }
        if (whole) {
          const uint32_t buf = my_staging + (uint32_t)(bi * STAGING_BYTES);
          if (lane == 0 && stores >= nbuf) {  // this buffer's previous store has read it
            if (nbuf == 2) bulk_wait_read<1>(); else bulk_wait_read<0>();
          }
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(buf + (uint32_t)(lane * 128) + ((uint32_t)(c ^ (lane & 7)) << 4), packed[c]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(mo, tl.nb * TN + ocol, tl.row0 + r0, buf);
            bulk_commit();
          }
          ++stores;
          if (++bi == nbuf) bi = 0;
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(optr + (size_t)(tl.row0 + r0 + lane) * NOUT + tl.nb * TN + ocol);
#pragma unroll
          for (int c = 0; c < 8; ++c) dst[c] = packed[c];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();  // every store has left shared memory and landed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
  }
}

// ---- CTA-pair kernel -------------------------------------------------------------------
// A cluster of two CTAs computes a 256-row x 256-column tile with tcgen05.mma.cta_group::2:
// each CTA holds its own 128 rows of A and half of the B rows, so each SM stages 32 KB per
// 64-wide k-block instead of 48 KB, and six stages fit.  The last rows of an expert, when
// 128 or fewer, form a half tile: an M = 128 pair MMA over 64 rows per CTA (measured TMEM
// layout: a CTA's 64 rows sit in lanes 0-63 for accumulator columns 0-127 and again in
// lanes 64-127 for columns 128-255), so no expert wastes more than 127 padded rows.
// GEMM1's B half of each CTA is [64 gate rows; the same 64 up rows] (one two-plane box), so
// every lane holds the gate and up values of the same outputs.  Each CTA issues its A
// copies from warp 6 and its B copies from warp 0 (two issuing warps keep the copy engine
// busier than one, measured); all copies count on the leader's full barrier.  The leader's
// warp 1 issues every MMA and releases a stage in both CTAs with one multicast commit; each
// CTA's epilogue warps drain their own TMEM lanes and arrive on the leader's
// accumulator-empty barrier.
namespace pair {
constexpr int PM = 256;                  // rows per pair tile
constexpr int HB = 128;                  // B rows per CTA
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB (8 KB used by a half tile)
constexpr int B_BYTES = HB * BK * 2;     // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 224;             // warps: 0 B copies, 1 MMA, 2-5 epilogue, 6 A copies
constexpr int STAGING_BYTES = 32 * 128;  // one 32-row x 64-column bf16 output block
constexpr uint32_t IDESC_FULL = idesc_bf16(PM, BN);
constexpr uint32_t IDESC_HALF = idesc_bf16(PM / 2, BN);
}  // namespace pair

// map_a / map_a_half: A with 128-row / 64-row boxes.  MODE 0: map_b is a two-plane gate/up
// map with a (64, 64, 2) box (b_planes 1: gate plane first, 2: up plane first) or, with
// b_planes 0, a 64-row gate map with map_b_up the matching up map.  MODE 1: map_b is W_down
// with a 128-row box.
template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::THREADS, 1)
pair_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_a_half,
                 const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b_up,
                 const __grid_constant__ CUtensorMap map_out, const int32_t* __restrict__ offsets, int G,
                 int M_total, int K, int NOUT, int b_planes, int nbuf, __nv_bfloat16* __restrict__ out,
                 int* __restrict__ status) {
  constexpr bool SWIGLU = MODE == 0;
  constexpr int TN = SWIGLU ? BN / 2 : BN;  // output columns per tile
  constexpr int S = pair::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // output staging: nbuf 4 KB buffers (32 rows x 64 bf16, 128-byte swizzle) per epilogue warp
  uint8_t* staging = smem + S * pair::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + 4 * nbuf * pair::STAGING_BYTES);
  // bars: full[S] (leader's are used), empty[S], tfull[2], tempty[2] (leader's), done
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* wtot = reinterpret_cast<int*>(tmem_holder + 2);  // [8]
  int* tile_start = wtot + 8;                            // [G + 1]

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int NB = (NOUT + TN - 1) / TN;
  const int KB = K / BK;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S + s); };
  auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * S + a); };
  auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * S + 2 + a); };
  const uint32_t done_bar = smem_u32(bars + 2 * S + 4);

  if (t == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 2);   // the leader's two copy-issuing threads; bytes of both CTAs
      mbar_init(empty_bar(s), 1);  // one multicast commit per use
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);  // four epilogue warps in each CTA of the pair
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // warp 1 of both CTAs allocates the pair's tensor memory together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
    if (SWIGLU && b_planes == 0)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b_up)) : "memory");
  }
  if (warp == 6 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a_half)) : "memory");
  }

  grid_dep_wait();  // set-up done; the offsets and operands come from earlier kernels
  grid_dep_launch();

  // tile_start[g] = sum over g' < g of (256-row blocks of g') * NB
  {
    const int per = (G + pair::THREADS - 1) / pair::THREADS;
    const int g0 = min(G, t * per), g1 = min(G, g0 + per);
    int local = 0;
    for (int g = g0; g < g1; ++g) {
      const int s0 = min(max(__ldg(offsets + g), 0), M_total);
      const int e0 = min(max(__ldg(offsets + g + 1), s0), M_total);
      local += ((e0 - s0 + pair::PM - 1) / pair::PM) * NB;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += wtot[w];
    base += incl - local;
    for (int g = g0; g < g1; ++g) {
      tile_start[g] = base;
      const int s0 = min(max(__ldg(offsets + g), 0), M_total);
      const int e0 = min(max(__ldg(offsets + g + 1), s0), M_total);
      base += ((e0 - s0 + pair::PM - 1) / pair::PM) * NB;
    }
    if (t == pair::THREADS - 1) {
      int tot = 0;
      for (int w = 0; w < pair::THREADS / 32; ++w) tot += wtot[w];
      tile_start[G] = tot;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and tensor memory exist before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total_tiles = tile_start[G];

  if ((warp == 0 || warp == 6) && lane == 0) {
    // ---------------- copy issue: warp 0 the B half, warp 6 the A rows ----------------
    const bool is_b = warp == 0;
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    for (int tile = pair_id; tile < total_tiles; tile += npairs) {
      const Tile tl = decode_rows<pair::PM>(tile, tile_start, G, offsets, M_total, NB);
      const bool half = tl.rows <= pair::PM / 2;
      const int a_row = tl.row0 + (int)rank * (half ? BM / 2 : BM);
      const int b_row = tl.g * NOUT + tl.nb * TN + (int)rank * (SWIGLU ? TN / 2 : pair::HB);
      const uint32_t tx = is_b ? 2 * pair::B_BYTES : 2 * (half ? pair::A_BYTES / 2 : pair::A_BYTES);
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status, true)) { ok = false; break; }
        const uint32_t dst = smem_u32(smem + stage * pair::STAGE_BYTES) + (is_b ? pair::A_BYTES : 0);
        const uint32_t lead_full = map_to_rank(full_bar(stage), 0);
        if (leader) mbar_expect_tx(full_bar(stage), tx);
        if (!is_b) {
          tma_load_2d_pair(dst, half ? &map_a_half : &map_a, kb * BK, a_row, lead_full);
        } else if (SWIGLU && b_planes != 0) {
          tma_load_3d_pair(dst, &map_b, kb * BK, b_row, 0, lead_full);
        } else if (SWIGLU) {
          tma_load_2d_pair(dst, &map_b, kb * BK, b_row, lead_full);
          tma_load_2d_pair(dst + pair::B_BYTES / 2, &map_b_up, kb * BK, b_row, lead_full);
        } else {
          tma_load_2d_pair(dst, &map_b, kb * BK, b_row, lead_full);
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    // every copy this thread issued has landed once the leader's MMA has released its stage
    for (int s = 0; s < S; ++s)
      if ((issued >> s) & 1u) mbar_wait(empty_bar(s), (issued_par >> s) & 1u, abort_flag, status, false);
  } else if (warp == 1) {
    if (lane == 0) {
      if (leader) {
        // ---------------- MMA issue (leader only) ----------------
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        for (int tile = pair_id; tile < total_tiles; tile += npairs) {
          const Tile tl = decode_rows<pair::PM>(tile, tile_start, G, offsets, M_total, NB);
          const uint32_t idesc = tl.rows <= pair::PM / 2 ? pair::IDESC_HALF : pair::IDESC_FULL;
          if (!mbar_wait_cluster(tempty_bar(acc), acc_phase ^ 1u, abort_flag, status, true)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          bool ok = true;
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(full_bar(stage), phase, abort_flag, status, true)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a_base = smem_u32(smem + stage * pair::STAGE_BYTES);
            const uint32_t b_base = a_base + pair::A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / UK; ++k)
              tc_mma_pair(d_tmem, sw128_desc(a_base + k * UK * 2), sw128_desc(b_base + k * UK * 2), idesc,
                          (kb | k) != 0 ? 1u : 0u);
            tc_commit_pair(empty_bar(stage), 0x3);
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          tc_commit_pair(tfull_bar(acc), 0x3);
          if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        // every pair MMA issued so far completes before either CTA frees its tensor memory
        tc_commit_pair(done_bar, 0x3);
      }
      mbar_wait(done_bar, 0, abort_flag, status, false);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
    // Each warp owns 32 rows of the tile and writes them in 64-column blocks: the block is
    // packed to bf16, staged in shared memory in the 128-byte swizzled layout and stored by
    // one TMA bulk store; a block that crosses the end of its expert's rows (the next
    // expert's rows follow in memory) is written row by row from registers instead.
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int tlane = q * 32 + lane;
    const uint32_t lead_tempty0 = map_to_rank(tempty_bar(0), 0), lead_tempty1 = map_to_rank(tempty_bar(1), 0);
    const int gate_first = b_planes != 2;  // plane order of each 64-row B block
    const uint32_t my_staging = smem_u32(staging) + (uint32_t)(q * nbuf * pair::STAGING_BYTES);
    int acc = 0, bi = 0, stores = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair_id; tile < total_tiles; tile += npairs) {
      const Tile tl = decode_rows<pair::PM>(tile, tile_start, G, offsets, M_total, NB);
      const bool half = tl.rows <= pair::PM / 2;
      const bool ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, status, true);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      // half tile: lanes 0-63 hold the CTA's 64 rows for accumulator columns 0-127, lanes
      // 64-127 the same rows for columns 128-255 (read back at TMEM columns 0-127)
      const int row = half ? (tlane & 63) : tlane;
      const int pr_base = (int)rank * (half ? BM / 2 : BM) + (row & ~31);  // first row of the warp
      const int pr = pr_base + lane;                                          // row within the tile
      const bool valid = pr < tl.rows;
      const bool whole = pr_base + 32 <= tl.rows;  // warp-uniform
      const int units = SWIGLU ? (half ? 1 : 2) : (half ? 2 : 4);
#pragma unroll 1
      for (int u = 0; u < units; ++u) {
        // accumulator columns of this 64-column block and its output columns in the tile
        int ocol;
        uint32_t c_a, c_b;  // SwiGLU: gate and up TMEM columns; down: TMEM column
        if (SWIGLU) {
          const int fb = half ? (tlane >> 6) : u;  // [leader gate|up 64+64][other CTA gate|up]
          const uint32_t cb = half ? 0u : (uint32_t)(fb * 128);
          c_a = cb + (gate_first ? 0u : 64u);
          c_b = cb + (gate_first ? 64u : 0u);
          ocol = fb * 64;
        } else {
          c_a = (uint32_t)(u * 64);
          c_b = 0;
          ocol = (half ? (tlane >> 6) * 128 : 0) + u * 64;
        }
        if (tl.nb * TN + ocol >= NOUT) continue;  // column tail (warp-uniform)
        uint4 packed[8];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (SWIGLU) {
            uint32_t gv[32], uv[32];
            tmem_ld32(taddr + c_a + c * 32, gv);
            tmem_ld32(taddr + c_b + c * 32, uv);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float h[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float g = __uint_as_float(gv[v * 8 + i]);
                const float uu = __uint_as_float(uv[v * 8 + i]);
                h[i] = __fdividef(g, 1.0f + __expf(-g)) * uu;
              }
              packed[c * 4 + v] = f32_to_bf16x8(h);
            }
          } else {
            uint32_t yv[32];
            tmem_ld32(taddr + c_a + c * 32, yv);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float y[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) y[i] = __uint_as_float(yv[v * 8 + i]);
              packed[c * 4 + v] = f32_to_bf16x8(y);
            }
          }
        }
        if (whole) {
          const uint32_t buf = my_staging + (uint32_t)(bi * pair::STAGING_BYTES);
          if (lane == 0 && stores >= nbuf) {  // this buffer's previous store has read it
            if (nbuf == 2) bulk_wait_read<1>(); else bulk_wait_read<0>();
          }
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(buf + (uint32_t)(lane * 128) + ((uint32_t)(c ^ (lane & 7)) << 4), packed[c]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&map_out, tl.nb * TN + ocol, tl.row0 + pr_base, buf);
            bulk_commit();
          }
          ++stores;
          if (++bi == nbuf) bi = 0;
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + (size_t)(tl.row0 + pr) * NOUT + tl.nb * TN + ocol);
#pragma unroll
          for (int c = 0; c < 8; ++c) dst[c] = packed[c];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(acc));
        else mbar_arrive_remote(acc == 0 ? lead_tempty0 : lead_tempty1);
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();  // every store has left shared memory and landed
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA frees tensor memory or exits while the pair still works
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
  }
}

// ---- host: tensor maps ---------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_planes_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t planes,
                          uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, planes};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One tensor map over both projections: planes {gate, up} (or {up, gate} when w_up lies
// below w_gate; *planes = 2) 'plane distance' bytes apart, so that a 3-D box of
// (64 columns, box_rows rows, 2 planes) brings the gate and up rows of a tile in one copy.
// Returns false (and the caller keeps two 2-D maps) if the driver rejects the layout.
bool make_map_gate_up(CUtensorMap* m, const void* w_gate, const void* w_up, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, int* planes) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uintptr_t g = reinterpret_cast<uintptr_t>(w_gate), u = reinterpret_cast<uintptr_t>(w_up);
  const uintptr_t lo = g < u ? g : u, dist = g < u ? u - g : g - u;
  if (dist < rows * cols * 2 || dist % 16 != 0 || dist >= (1ULL << 40)) return false;
  cuuint64_t dims[3] = {cols, rows, 2};
  cuuint64_t strides[2] = {cols * 2, (cuuint64_t)dist};
  cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, reinterpret_cast<void*>(lo), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  *planes = g < u ? 1 : 2;
  return true;
}

size_t smem_bytes(int G, int nbuf) {
  return 1024 + (size_t)STAGES * STAGE_BYTES + (size_t)4 * nbuf * STAGING_BYTES + 256 + (size_t)(G + 32) * 4;
}

// The extra group of a launch (the shared expert's tiles in the routed experts' launch): its
// A rows, B weights (b_planes as for the routed B) and output, M rows; M = 0: none.
struct ExtraGroup {
  const CUtensorMap* a = nullptr;
  const CUtensorMap* b = nullptr;
  const CUtensorMap* out_map = nullptr;
  int M = 0;
  void* out = nullptr;
  int b_planes = 0;
};

template <int MODE>
moe_status_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& out_map,
                    const int32_t* offsets, int G, int M_total, int K, int NOUT, void* out, int* status,
                    cudaStream_t s, const void* xg = nullptr, int NX = 0, const int32_t* perm = nullptr,
                    int b_planes = 0, const ExtraGroup& x = ExtraGroup()) {
  const int nbuf = smem_bytes(G, 2) <= 227 * 1024 ? 2 : 1;  // double-buffer the staging if it fits
  const size_t smem = smem_bytes(G, nbuf);
  auto kern = grouped_gemm_kernel<MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int TN = MODE != 1 ? BN / 2 : BN;
  const long long NB = (NOUT + TN - 1) / TN;
  const int M2 = x.M;
  const long long max_tiles = ((long long)(M_total + BM - 1) / BM + G) * NB + ((long long)(M2 + BM - 1) / BM) * NB;
  const int grid = (int)std::min<long long>(max_tiles, (long long)cta_cap());
  return launch_kernel(kern, dim3(grid), dim3(kThreads<MODE>), smem, s, a, b0, b1, out_map, offsets, G, M_total, K,
                       NOUT, static_cast<__nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(xg), NX, perm,
                       b_planes, nbuf, status, M2 > 0 ? *x.a : a, M2 > 0 ? *x.b : b0, M2 > 0 ? *x.out_map : out_map,
                       M2, static_cast<__nv_bfloat16*>(M2 > 0 ? x.out : out), x.b_planes);
}

size_t pair_smem_bytes(int G, int nbuf) {
  return 1024 + (size_t)pair::STAGES * pair::STAGE_BYTES + (size_t)4 * nbuf * pair::STAGING_BYTES + 256 +
         (size_t)(G + 16) * 4;
}

template <int MODE>
moe_status_t launch_pair(const CUtensorMap& a, const CUtensorMap& a_half, const CUtensorMap& b,
                         const CUtensorMap& b_up, const CUtensorMap& out_map, int b_planes, const int32_t* offsets,
                         int G, int M_total, int K, int NOUT, void* out, int* status, cudaStream_t s) {
  const int nbuf = pair_smem_bytes(G, 2) <= 227 * 1024 ? 2 : 1;  // double-buffer the staging if it fits
  const size_t smem = pair_smem_bytes(G, nbuf);
  auto kern = pair_gemm_kernel<MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int TN = MODE == 0 ? BN / 2 : BN;
  const long long NB = (NOUT + TN - 1) / TN;
  const long long max_tiles = ((long long)(M_total + pair::PM - 1) / pair::PM + G) * NB;
  const int pairs = (int)std::min<long long>(max_tiles, (long long)(cta_cap() / 2));
  return launch_kernel(kern, dim3(2 * pairs), dim3(pair::THREADS), smem, s, a, a_half, b, b_up, out_map, offsets, G,
                       M_total, K, NOUT, b_planes, nbuf, static_cast<__nv_bfloat16*>(out), status);
}

}  // namespace tc

namespace simt {

// fp32 grouped SwiGLU on CUDA cores: 32 x 64 output tiles, 256 threads with 2 x 4 outputs
// each (two rows of four columns: a small layer still gets several warps per SM), 32-wide K
// slices staged in shared memory (k-major, so a thread reads its two rows as one float2 and
// four columns as one float4), the next slice loaded into registers during the FMAs.  Every
// output is one fp32 FMA chain over K in index order (bit-identical to a plain dot-product
// loop).  Tiles are (group, 32-row block, column block); a CTA finds its group by walking
// the offsets.
constexpr int TM = 32, TN = 64, TK = 32, PAD = 4;

struct SimtTile {
  int g, row0, rows, col0;
  bool valid;
};

__device__ __forceinline__ SimtTile simt_tile(int t, const int32_t* __restrict__ offsets, int G, int M, int CB) {
  SimtTile r{0, 0, 0, 0, false};
  int base = 0;
  for (int g = 0; g < G; ++g) {
    const int s = min(max(offsets[g], 0), M);
    const int e = min(max(offsets[g + 1], s), M);
    const int n = ((e - s + TM - 1) / TM) * CB;
    if (t < base + n) {
      const int local = t - base;
      const int rb = local / CB;
      r.g = g;
      r.row0 = s + rb * TM;
      r.rows = min(TM, e - r.row0);
      r.col0 = (local - rb * CB) * TN;
      r.valid = true;
      return r;
    }
    base += n;
  }
  return r;
}

// One thread's share of a ROWS-row x TK-column slice of a row-major [*, ld] matrix (rows
// [row0, row0 + rows), columns [k0, k0 + TK); zero beyond `rows`): ROWS * TK / 4 / 256 float4.
template <int ROWS>
struct Slice {
  static constexpr int V = ROWS * TK / 4 / 256;
  float4 v[V];
  __device__ __forceinline__ void load(const float* __restrict__ src, int ld, int row0, int rows, int k0) {
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int i = threadIdx.x + q * 256;
      const int m = i / (TK / 4), kq = (i % (TK / 4)) * 4;
      v[q] = m < rows ? *reinterpret_cast<const float4*>(src + (size_t)(row0 + m) * ld + k0 + kq)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // into dst[k][m] (k-major, so the compute loop reads rows or columns as one vector)
  __device__ __forceinline__ void store(float (*dst)[ROWS + PAD]) const {
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int i = threadIdx.x + q * 256;
      const int m = i / (TK / 4), kq = (i % (TK / 4)) * 4;
      dst[kq + 0][m] = v[q].x;
      dst[kq + 1][m] = v[q].y;
      dst[kq + 2][m] = v[q].z;
      dst[kq + 3][m] = v[q].w;
    }
  }
};

// H[r, f] = SiLU(x_r . W_gate[g, f]) * (x_r . W_up[g, f]).  The next K slice is loaded into
// registers while the current one is multiplied out of shared memory.
__global__ void __launch_bounds__(256, 2) swiglu_up_kernel(const float* __restrict__ x, const int32_t* __restrict__ offsets,
                                                        int G, int M, int D, int F, const float* __restrict__ wg,
                                                        const float* __restrict__ wu, float* __restrict__ h) {
  __shared__ __align__(16) float xs[TK][TM + PAD], gs[TK][TN + PAD], us[TK][TN + PAD];
  grid_dep_wait();
  grid_dep_launch();
  const int CB = (F + TN - 1) / TN;
  const SimtTile tl = simt_tile(blockIdx.x, offsets, G, M, CB);
  if (!tl.valid) return;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int ncols = min(TN, F - tl.col0);
  const float* wgg = wg + ((size_t)tl.g * F + tl.col0) * D;
  const float* wug = wu + ((size_t)tl.g * F + tl.col0) * D;
  float ag[2][4] = {}, au[2][4] = {};
  Slice<TM> sx;
  Slice<TN> sg, su;
  sx.load(x, D, tl.row0, tl.rows, 0);
  sg.load(wgg, D, 0, ncols, 0);
  su.load(wug, D, 0, ncols, 0);
  for (int k0 = 0; k0 < D; k0 += TK) {
    sx.store(xs);
    sg.store(gs);
    su.store(us);
    __syncthreads();
    if (k0 + TK < D) {  // next slice in flight during the FMAs
      sx.load(x, D, tl.row0, tl.rows, k0 + TK);
      sg.load(wgg, D, 0, ncols, k0 + TK);
      su.load(wug, D, 0, ncols, k0 + TK);
    }
#pragma unroll 8
    for (int k = 0; k < TK; ++k) {
      const float2 a = *reinterpret_cast<const float2*>(&xs[k][ty * 2]);
      const float4 b = *reinterpret_cast<const float4*>(&gs[k][tx * 4]);
      const float4 c = *reinterpret_cast<const float4*>(&us[k][tx * 4]);
      const float av[2] = {a.x, a.y}, bv[4] = {b.x, b.y, b.z, b.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ag[i][j] = fmaf(av[i], bv[j], ag[i][j]);
          au[i][j] = fmaf(av[i], cv[j], au[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = ty * 2 + i;
    if (r >= tl.rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = tx * 4 + j;
      if (c < ncols) {
        const float a = ag[i][j];
        h[(size_t)(tl.row0 + r) * F + tl.col0 + c] = (a / (1.0f + expf(-a))) * au[i][j];
      }
    }
  }
}

// Y[r, d] = H_r . W_down[g, d]
__global__ void __launch_bounds__(256, 2) swiglu_down_kernel(const float* __restrict__ h, const int32_t* __restrict__ offsets,
                                                          int G, int M, int D, int F, const float* __restrict__ wd,
                                                          float* __restrict__ y) {
  __shared__ __align__(16) float hs[TK][TM + PAD], ds[TK][TN + PAD];
  grid_dep_wait();
  grid_dep_launch();
  const int CB = (D + TN - 1) / TN;
  const SimtTile tl = simt_tile(blockIdx.x, offsets, G, M, CB);
  if (!tl.valid) return;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int ncols = min(TN, D - tl.col0);
  const float* wdg = wd + ((size_t)tl.g * D + tl.col0) * F;
  float acc[2][4] = {};
  Slice<TM> sh;
  Slice<TN> sd;
  sh.load(h, F, tl.row0, tl.rows, 0);
  sd.load(wdg, F, 0, ncols, 0);
  for (int k0 = 0; k0 < F; k0 += TK) {
    sh.store(hs);
    sd.store(ds);
    __syncthreads();
    if (k0 + TK < F) {
      sh.load(h, F, tl.row0, tl.rows, k0 + TK);
      sd.load(wdg, F, 0, ncols, k0 + TK);
    }
#pragma unroll 8
    for (int k = 0; k < TK; ++k) {
      const float2 a = *reinterpret_cast<const float2*>(&hs[k][ty * 2]);
      const float4 b = *reinterpret_cast<const float4*>(&ds[k][tx * 4]);
      const float av[2] = {a.x, a.y}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = ty * 2 + i;
    if (r >= tl.rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = tx * 4 + j;
      if (c < ncols) y[(size_t)(tl.row0 + r) * D + tl.col0 + c] = acc[i][j];
    }
  }
}

}  // namespace simt
}  // namespace moe

namespace moe {
namespace tc {
// CTA-pair tiles (256 rows) pay off when experts average at least two 128-row blocks; the
// MOE_GROUPED_GEMM environment variable ("pair", "single", anything else = automatic)
// overrides the choice.
bool use_pair(int G, int M_total) {
  if (cta_cap() < 2) return false;
  const char* e = std::getenv("MOE_GROUPED_GEMM");
  if (e && std::strcmp(e, "pair") == 0) return true;
  if (e && std::strcmp(e, "single") == 0) return false;
  return (long long)M_total >= 256LL * G;
}
}  // namespace tc
}  // namespace moe

extern "C" moe_status_t moe_grouped_swiglu(const void* x_perm, moe_dtype_t dtype, const int32_t* offsets,
                                           int G, int M_total, int D, int F, const void* w_gate,
                                           const void* w_up, const void* w_down, void* h_workspace,
                                           void* y_perm, moe_stream_t stream) {
  using namespace moe;
  if (G < 1 || M_total < 0 || D <= 0 || F <= 0) return MOE_ERR_INVALID_ARG;
  if (D % 64 != 0 || F % 64 != 0 || G > tc::MAX_GROUPS) return MOE_ERR_UNSUPPORTED;
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if ((long long)G * F >= (1LL << 31) || (long long)G * D >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (M_total == 0) return MOE_OK;
  if (!x_perm || !offsets || !w_gate || !w_up || !w_down || !h_workspace || !y_perm)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(h_workspace) || !aligned16(y_perm))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_cuda(stream);
  if (dtype == MOE_F32) {
    // at most (row blocks of M_total + one partial block per group) x column blocks tiles
    const long long rb = (M_total + simt::TM - 1) / simt::TM + G;
    const long long t1 = rb * ((F + simt::TN - 1) / simt::TN), t2 = rb * ((D + simt::TN - 1) / simt::TN);
    if (t1 >= (1LL << 31) || t2 >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    const moe_status_t st = launch_kernel(
        simt::swiglu_up_kernel, dim3((unsigned)t1), dim3(256), 0, s, static_cast<const float*>(x_perm), offsets, G,
        M_total, D, F, static_cast<const float*>(w_gate), static_cast<const float*>(w_up),
        static_cast<float*>(h_workspace));
    if (st != MOE_OK) return st;
    return launch_kernel(simt::swiglu_down_kernel, dim3((unsigned)t2), dim3(256), 0, s,
                         static_cast<const float*>(h_workspace), offsets, G, M_total, D, F,
                         static_cast<const float*>(w_down), static_cast<float*>(y_perm));
  }
  int* status = device_status_word();
  if (!status) return MOE_ERR_CUDA;
  if (tc::use_pair(G, M_total)) {
    CUtensorMap ma, ma2, mg, mu, mh, mh2, md, mgu, mho, myo;
    if (!tc::make_map_bf16(&mho, h_workspace, (uint64_t)M_total, (uint64_t)F, 32) ||
        !tc::make_map_bf16(&myo, y_perm, (uint64_t)M_total, (uint64_t)D, 32) ||
        !tc::make_map_bf16(&ma, x_perm, (uint64_t)M_total, (uint64_t)D, tc::BM) ||
        !tc::make_map_bf16(&ma2, x_perm, (uint64_t)M_total, (uint64_t)D, tc::BM / 2) ||
        !tc::make_map_bf16(&mh, h_workspace, (uint64_t)M_total, (uint64_t)F, tc::BM) ||
        !tc::make_map_bf16(&mh2, h_workspace, (uint64_t)M_total, (uint64_t)F, tc::BM / 2) ||
        !tc::make_map_bf16(&md, w_down, (uint64_t)G * D, (uint64_t)F, tc::pair::HB))
      return MOE_ERR_CUDA;
    int planes = 0;
    moe_status_t st;
    if (tc::make_map_gate_up(&mgu, w_gate, w_up, (uint64_t)G * F, (uint64_t)D, tc::BN / 4, &planes)) {
      st = tc::launch_pair<0>(ma, ma2, mgu, mgu, mho, planes, offsets, G, M_total, D, F, h_workspace, status, s);
    } else {
      if (!tc::make_map_bf16(&mg, w_gate, (uint64_t)G * F, (uint64_t)D, tc::BN / 4) ||
          !tc::make_map_bf16(&mu, w_up, (uint64_t)G * F, (uint64_t)D, tc::BN / 4))
        return MOE_ERR_CUDA;
      st = tc::launch_pair<0>(ma, ma2, mg, mu, mho, 0, offsets, G, M_total, D, F, h_workspace, status, s);
    }
    if (st != MOE_OK) return st;
    return tc::launch_pair<1>(mh, mh2, md, md, myo, 0, offsets, G, M_total, F, D, y_perm, status, s);
  }
  CUtensorMap ma, mg, mu, mh, md, mho, myo;
  if (!tc::make_map_bf16(&ma, x_perm, (uint64_t)M_total, (uint64_t)D, tc::A_BOX) ||
      !tc::make_map_bf16(&mg, w_gate, (uint64_t)G * F, (uint64_t)D, tc::BN / 2) ||
      !tc::make_map_bf16(&mu, w_up, (uint64_t)G * F, (uint64_t)D, tc::BN / 2) ||
      !tc::make_map_bf16(&mh, h_workspace, (uint64_t)M_total, (uint64_t)F, tc::A_BOX) ||
      !tc::make_map_bf16(&md, w_down, (uint64_t)G * D, (uint64_t)F, tc::BN) ||
      !tc::make_map_bf16(&mho, h_workspace, (uint64_t)M_total, (uint64_t)F, 32) ||
      !tc::make_map_bf16(&myo, y_perm, (uint64_t)M_total, (uint64_t)D, 32))
    return MOE_ERR_CUDA;
  CUtensorMap mgu;
  int planes = 0;
  const bool gu = tc::make_map_gate_up(&mgu, w_gate, w_up, (uint64_t)G * F, (uint64_t)D, tc::BN / 2, &planes);
  moe_status_t st = gu ? tc::launch<0>(ma, mgu, mgu, mho, offsets, G, M_total, D, F, h_workspace, status, s,
                                       nullptr, 0, nullptr, planes)
                       : tc::launch<0>(ma, mg, mu, mho, offsets, G, M_total, D, F, h_workspace, status, s);
  if (st != MOE_OK) return st;
  return tc::launch<1>(mh, md, md, myo, offsets, G, M_total, F, D, y_perm, status, s);
}

extern "C" moe_status_t moe_grouped_swiglu_ex(const void* x_perm, moe_dtype_t dtype, const int32_t* offsets,
                                              int G, int M_total, int D, int F, const void* w_gate,
                                              const void* w_up, const void* w_down, void* h_workspace,
                                              void* y_perm, int max_ctas, moe_stream_t stream) {
  if (max_ctas < 0) return MOE_ERR_INVALID_ARG;
  const int saved = moe::tc::g_max_ctas;
  moe::tc::g_max_ctas = max_ctas;
  const moe_status_t st = moe_grouped_swiglu(x_perm, dtype, offsets, G, M_total, D, F, w_gate, w_up, w_down,
                                             h_workspace, y_perm, stream);
  moe::tc::g_max_ctas = saved;
  return st;
}

namespace moe {
namespace {
// moe_grouped_swiglu_shared; with h_ready, hs_workspace already holds the shared expert's H
// (made by the router launch) and only its second GEMM runs, in the routed GEMM2 launch.
moe_status_t grouped_shared_impl(const void* x_perm, const int32_t* perm_token, const int32_t* offsets, int G,
                                 int M_total, int D, int F, const void* w_gate, const void* w_up,
                                 const void* w_down, void* h_workspace, void* y_perm, const void* xn, int N,
                                 const void* ws_gate, const void* ws_up, const void* ws_down, void* hs_workspace,
                                 void* shared_y, moe_stream_t stream, bool h_ready) {
  const bool gather = perm_token != nullptr;  // routed rows read from xn through perm_token
  if (G < 1 || M_total < 0 || D <= 0 || F <= 0 || N < 0) return MOE_ERR_INVALID_ARG;
  if (D % 64 != 0 || F % 64 != 0 || G > tc::MAX_GROUPS) return MOE_ERR_UNSUPPORTED;
  if ((long long)G * F >= (1LL << 31) || (long long)G * D >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (M_total > 0 && ((!gather && !x_perm) || !offsets || !w_gate || !w_up || !w_down || !h_workspace || !y_perm))
    return MOE_ERR_INVALID_ARG;
  if (gather && M_total > 0 && (!xn || N < 1)) return MOE_ERR_INVALID_ARG;
  if (N > 0 && (!ws_down || !hs_workspace || !shared_y || (!h_ready && (!xn || !ws_gate || !ws_up))))
    return MOE_ERR_INVALID_ARG;
  for (const void* p : {x_perm, (const void*)w_gate, w_up, w_down, (const void*)h_workspace, (const void*)y_perm, xn,
                        ws_gate, ws_up, ws_down, (const void*)hs_workspace, (const void*)shared_y})
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  auto routed_alone = [&]() {
    return gather ? moe_grouped_swiglu_gather(xn, N, perm_token, offsets, G, M_total, D, F, w_gate, w_up, w_down,
                                              h_workspace, y_perm, stream)
                  : moe_grouped_swiglu(x_perm, MOE_BF16, offsets, G, M_total, D, F, w_gate, w_up, w_down,
                                       h_workspace, y_perm, stream);
  };
  if (N == 0) return routed_alone();
  if (!offsets) return MOE_ERR_INVALID_ARG;
  // Routed experts large enough for CTA pairs run on the pair kernels first; the shared
  // expert then runs alone as the extra group of one-CTA launches with no routed rows.
  const bool separate = M_total == 0 || tc::use_pair(G, M_total);
  if (separate && M_total > 0) {
    const moe_status_t st = routed_alone();
    if (st != MOE_OK) return st;
  }
  const int Mr = separate ? 0 : M_total;  // routed rows in these launches
  int* status = device_status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = as_cuda(stream);
  CUtensorMap ma, mg, mu, mh, md, mho, myo, mgu;
  CUtensorMap xa, xgu, xh, xd, xho, xyo;
  int planes = 0, xplanes = 0;
  if (!tc::make_map_bf16(&xh, hs_workspace, (uint64_t)N, (uint64_t)F, tc::A_BOX) ||
      !tc::make_map_bf16(&xd, ws_down, (uint64_t)D, (uint64_t)F, tc::BN) ||
      !tc::make_map_bf16(&xho, hs_workspace, (uint64_t)N, (uint64_t)F, 32) ||
      !tc::make_map_bf16(&xyo, shared_y, (uint64_t)N, (uint64_t)D, 32))
    return MOE_ERR_CUDA;
  if (!h_ready) {  // the shared expert's first GEMM runs here too
    if (!tc::make_map_bf16(&xa, xn, (uint64_t)N, (uint64_t)D, tc::A_BOX)) return MOE_ERR_CUDA;
    if (!tc::make_map_gate_up(&xgu, ws_gate, ws_up, (uint64_t)F, (uint64_t)D, tc::BN / 2, &xplanes))
      return MOE_ERR_UNSUPPORTED;  // the shared gate/up pair must form one two-plane map
  }
  bool gu = false;
  if (Mr > 0) {
    if (!tc::make_map_bf16(&ma, gather ? xn : x_perm, (uint64_t)(gather ? N : Mr), (uint64_t)D, tc::A_BOX) ||
        !tc::make_map_bf16(&mg, w_gate, (uint64_t)G * F, (uint64_t)D, tc::BN / 2) ||
        !tc::make_map_bf16(&mu, w_up, (uint64_t)G * F, (uint64_t)D, tc::BN / 2) ||
        !tc::make_map_bf16(&mh, h_workspace, (uint64_t)Mr, (uint64_t)F, tc::A_BOX) ||
        !tc::make_map_bf16(&md, w_down, (uint64_t)G * D, (uint64_t)F, tc::BN) ||
        !tc::make_map_bf16(&mho, h_workspace, (uint64_t)Mr, (uint64_t)F, 32) ||
        !tc::make_map_bf16(&myo, y_perm, (uint64_t)Mr, (uint64_t)D, 32))
      return MOE_ERR_CUDA;
    gu = tc::make_map_gate_up(&mgu, w_gate, w_up, (uint64_t)G * F, (uint64_t)D, tc::BN / 2, &planes);
  } else {  // no routed tiles: the shared expert's maps stand in for the unused routed ones
    mh = xh; md = xd; mho = xho; myo = xyo;
    if (!h_ready) {
      ma = xa; mgu = xgu; mg = xgu; mu = xgu;
      gu = true;
      planes = xplanes;
    }
  }
  tc::ExtraGroup x1;
  if (!h_ready) {
    x1.a = &xa; x1.b = &xgu; x1.out_map = &xho; x1.M = N; x1.out = hs_workspace; x1.b_planes = xplanes;
  }
  moe_status_t st = MOE_OK;
  if (h_ready && Mr == 0)
    ;  // nothing left for a first GEMM
  else if (gather && Mr > 0)  // GEMM1 gathers the routed rows through perm_token and the shared rows in order
    st = gu ? tc::launch<2>(mgu, mgu, mgu, mho, offsets, G, Mr, D, F, h_workspace, status, s, xn, N, perm_token,
                            planes, x1)
            : tc::launch<2>(mg, mg, mu, mho, offsets, G, Mr, D, F, h_workspace, status, s, xn, N, perm_token, 0, x1);
  else
    st = gu ? tc::launch<0>(ma, mgu, mgu, mho, offsets, G, Mr, D, F, h_workspace, status, s, nullptr, 0, nullptr,
                            planes, x1)
            : tc::launch<0>(ma, mg, mu, mho, offsets, G, Mr, D, F, h_workspace, status, s, nullptr, 0, nullptr, 0, x1);
  if (st != MOE_OK) return st;
  tc::ExtraGroup x2;
  x2.a = &xh; x2.b = &xd; x2.out_map = &xyo; x2.M = N; x2.out = shared_y; x2.b_planes = 0;
  return tc::launch<1>(mh, md, md, myo, offsets, G, Mr, F, D, y_perm, status, s, nullptr, 0, nullptr, 0, x2);
}
}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_grouped_swiglu_shared(const void* x_perm, const int32_t* perm_token,
                                                  const int32_t* offsets, int G, int M_total, int D, int F,
                                                  const void* w_gate, const void* w_up, const void* w_down,
                                                  void* h_workspace, void* y_perm, const void* xn, int N,
                                                  const void* ws_gate, const void* ws_up, const void* ws_down,
                                                  void* hs_workspace, void* shared_y, moe_stream_t stream) {
  return moe::grouped_shared_impl(x_perm, perm_token, offsets, G, M_total, D, F, w_gate, w_up, w_down, h_workspace,
                                  y_perm, xn, N, ws_gate, ws_up, ws_down, hs_workspace, shared_y, stream, false);
}

extern "C" moe_status_t moe_grouped_swiglu_shared_h(const void* x_perm, const int32_t* perm_token,
                                                    const int32_t* offsets, int G, int M_total, int D, int F,
                                                    const void* w_gate, const void* w_up, const void* w_down,
                                                    void* h_workspace, void* y_perm, const void* xn, int N,
                                                    const void* ws_down, void* hs_workspace, void* shared_y,
                                                    moe_stream_t stream) {
  return moe::grouped_shared_impl(x_perm, perm_token, offsets, G, M_total, D, F, w_gate, w_up, w_down, h_workspace,
                                  y_perm, xn, N, nullptr, nullptr, ws_down, hs_workspace, shared_y, stream, true);
}

extern "C" moe_status_t moe_grouped_swiglu_gather(const void* xn, int N, const int32_t* perm_token,
                                                  const int32_t* offsets, int G, int M_total, int D, int F,
                                                  const void* w_gate, const void* w_up, const void* w_down,
                                                  void* h_workspace, void* y_perm, moe_stream_t stream) {
  using namespace moe;
  if (G < 1 || M_total < 0 || D <= 0 || F <= 0 || N < 0) return MOE_ERR_INVALID_ARG;
  if (D % 64 != 0 || F % 64 != 0 || G > tc::MAX_GROUPS) return MOE_ERR_UNSUPPORTED;
  if ((long long)G * F >= (1LL << 31) || (long long)G * D >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (M_total == 0) return MOE_OK;
  if (N == 0) return MOE_ERR_INVALID_ARG;  // rows to gather from, but no tokens
  if (!xn || !perm_token || !offsets || !w_gate || !w_up || !w_down || !h_workspace || !y_perm)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(xn) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(h_workspace) || !aligned16(y_perm))
    return MOE_ERR_INVALID_ARG;
  int* status = device_status_word();
  if (!status) return MOE_ERR_CUDA;
  cudaStream_t s = as_cuda(stream);
  CUtensorMap mg, mu, mh, md, mho, myo;
  const bool pair2 = tc::use_pair(G, M_total);  // GEMM2 on CTA pairs (128-row H boxes) or one CTA
  if (!tc::make_map_bf16(&mg, w_gate, (uint64_t)G * F, (uint64_t)D, tc::BN / 2) ||
      !tc::make_map_bf16(&mu, w_up, (uint64_t)G * F, (uint64_t)D, tc::BN / 2) ||
      !tc::make_map_bf16(&mh, h_workspace, (uint64_t)M_total, (uint64_t)F, pair2 ? tc::BM : tc::A_BOX) ||
      !tc::make_map_bf16(&md, w_down, (uint64_t)G * D, (uint64_t)F, tc::BN) ||
      !tc::make_map_bf16(&mho, h_workspace, (uint64_t)M_total, (uint64_t)F, 32) ||
      !tc::make_map_bf16(&myo, y_perm, (uint64_t)M_total, (uint64_t)D, 32))
    return MOE_ERR_CUDA;
  CUtensorMap mgu;
  int planes = 0;
  const bool gu = tc::make_map_gate_up(&mgu, w_gate, w_up, (uint64_t)G * F, (uint64_t)D, tc::BN / 2, &planes);
  moe_status_t st = gu ? tc::launch<2>(mgu, mgu, mgu, mho, offsets, G, M_total, D, F, h_workspace, status, s, xn,
                                       N, perm_token, planes)
                       : tc::launch<2>(mg, mg, mu, mho, offsets, G, M_total, D, F, h_workspace, status, s, xn, N,
                                       perm_token);
  if (st != MOE_OK) return st;
  if (pair2) {  // GEMM2 reads H, not gathered rows: CTA pairs as in moe_grouped_swiglu
    CUtensorMap mh2, mdp;
    if (!tc::make_map_bf16(&mh2, h_workspace, (uint64_t)M_total, (uint64_t)F, tc::BM / 2) ||
        !tc::make_map_bf16(&mdp, w_down, (uint64_t)G * D, (uint64_t)F, tc::pair::HB))
      return MOE_ERR_CUDA;
    return tc::launch_pair<1>(mh, mh2, mdp, mdp, myo, 0, offsets, G, M_total, F, D, y_perm, status, s);
  }
  return tc::launch<1>(mh, md, md, myo, offsets, G, M_total, F, D, y_perm, status, s);
}

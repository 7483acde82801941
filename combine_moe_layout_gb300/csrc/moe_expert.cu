// Expert stage between dispatch and combine: every expert's packed bf16 rows go
// through linear 1 with SwiGLU and then linear 2, on the 5th-generation tensor
// cores (tcgen05.mma with the accumulator in tensor memory, operands staged by
// TMA).
//
// "How GPUs Talk to Each Other During LLM Inference", section 7 (Mega MoE):
// between dispatch and combine every expert applies linear 1, SwiGLU and
// linear 2 to the tokens it received. Perplexity, "Efficient and portable
// mixture-of-experts communication", section "Dispatch": the receive side packs
// each expert's tokens contiguously so that they feed a grouped GEMM. The packed
// rows of expert e are rows [off[e*R], off[(e+1)*R]) of the buffers the receive
// hook writes, and one grouped-GEMM kernel runs each linear map:
//
//   gate/up:  h[p][i] = bf16( silu(x_p . w_gate[e][i]) * (x_p . w_up[e][i]) )
//   down:     y[p][j] = bf16( h_p . w_down[e][j] )
//
// bf16 operands, fp32 accumulation, silu(g) = g / (1 + exp(-g)) in fp32.
//
// Two kernels share the scheme below: grouped_gemm_kernel (one CTA per tile,
// M = 128) and grouped_gemm_pair_kernel (a cluster of two CTAs per tile,
// M = 256 with tcgen05 cta_group::2), taken for linear 2 of experts that
// average at least 512 rows.
//
// Kernel shape: one persistent CTA per SM, 192 threads.
//   warp 0      TMA producer: per 64-wide K block, a 128-row A tile and a
//               256-row (or 128-row) B tile, 128-byte swizzle, into a 4-stage
//               shared-memory ring.
//   warp 1      owns 512 TMEM columns (two 128 x 256 fp32 accumulators, so the
//               epilogue of one tile overlaps the MMAs of the next) and issues
//               tcgen05.mma (M = 128, N = 256 or 128, K = 16) from one lane.
//   warps 2-5   epilogue: each warp reads its 32-lane quarter of the
//               accumulator with tcgen05.ld, applies SwiGLU or plain bf16
//               rounding and stores the rows that belong to the tile's expert.
// A tile is up to 128 consecutive packed rows of one expert. For gate/up its
// 256 accumulator columns are 128 gate rows i0..i0+127 of the expert's weights
// followed by the 128 up rows of the same i, so SwiGLU pairs columns c and
// c + 128 of a thread's own row. Tiles are numbered expert by expert within two
// classes, interleaved (see tile_of): experts with several m-tiles and experts
// with one. Inside an expert they go in groups of G n-tiles, each group swept
// m-tile by m-tile with its G n-tiles innermost. The CTAs running at one time
// then share both the group's weight tiles and each m-tile of rows (read once
// per group instead of once per n-tile); G balances the two (see group_width).
//
// Every wait is bounded: a timeout records MOE_ETIMEOUT, every role of the CTA
// stops, the loads and MMAs already issued are waited for (again bounded) and
// the tensor memory is freed before the CTA exits.
#include <cuda_bf16.h>

#include <cmath>

#include "moe_tc.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;            // rows of a tile (tcgen05 M)
constexpr int kBK = 64;             // K elements per stage: one 128-byte swizzled row
constexpr int kUK = 16;             // K of one tcgen05.mma kind::f16
constexpr int kBNMax = 256;         // accumulator columns of a tile
constexpr int kStages = 4;
constexpr int kTileA = kBM * kBK * 2;
constexpr int kTileB = kBNMax * kBK * 2;
constexpr int kStage = kTileA + kTileB;
constexpr int kBoxBytes = kBoxRows * kBK * 2;
constexpr int kGemmThreads = 192;
constexpr uint32_t kTmemCols = 2 * kBNMax;
constexpr int kSmemFixed = 1024 + kStages * kStage + (2 * kStages + 5) * 8 + 8;
constexpr int kSmemMax = 227 * 1024;
// Width G of an n-tile group. The C tiles that run at one time cover about C/G
// m-tiles of rows (a bytes each) and G weight tiles (b bytes each); the bytes
// they touch, (C/G) a + G b, are least at G = sqrt(C a / b), capped so that the
// group's weight tiles stay well inside L2 while the group sweeps the rows.
// MOE_GEMM_GROUP_N > 0 fixes G instead.
#ifndef MOE_GEMM_GROUP_N
#define MOE_GEMM_GROUP_N 0
#endif
#ifndef MOE_GEMM_L2_GROUP_BYTES
#define MOE_GEMM_L2_GROUP_BYTES (64ll << 20)
#endif

static_assert(kTileA % 1024 == 0 && kStage % 1024 == 0 && kBoxBytes % 1024 == 0, "tiles on 1024-byte boundaries");
static_assert(kBK * 2 == 128, "one K block is one 128-byte swizzle row");
static_assert(kSmemFixed + 8 * 2 <= kSmemMax, "");

struct GemmArgs {
  const int32_t *region_offsets;  // [E*R + 1] packed-row offsets of the (expert, source rank) regions
  int32_t *err;
  __nv_bfloat16 *out;             // [rows][n_total]
  int rows;                       // rows of A and of out
  int E, R;
  int K;                          // contraction length: a multiple of 64
  int n_total;                    // output columns of a row (I for gate/up, H for down)
  int b_rows;                     // weight rows in one B tile: 256 (two boxes) or 128 (one box)
  int out_cols;                   // output columns of one tile: 128 (gate/up) or b_rows (down)
  int ntiles_n;                   // n_total / out_cols
  int expert_rows;                // weight rows of one expert in the tensor maps (I or H)
  int swiglu;                     // 1: gate/up tile with the SwiGLU epilogue
  int group_n;                    // n-tiles per group of the tile order (>= 1)
};

// bf16 epilogue of one 32-column chunk of a thread's accumulator row: SwiGLU
// over gate columns g[0..31] and up columns u[0..31], or plain rounding of
// r[0..31]; 64 bytes stored at dst.
__device__ __forceinline__ void store16(uint4 *d, uint4 v) { *d = v; }

__device__ __forceinline__ void store_swiglu32(__nv_bfloat16 *dst, const uint32_t (&r)[64]) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float g0 = __uint_as_float(r[2 * i]), g1 = __uint_as_float(r[2 * i + 1]);
    const float u0 = __uint_as_float(r[32 + 2 * i]), u1 = __uint_as_float(r[32 + 2 * i + 1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(g0 / (1.0f + expf(-g0)) * u0, g1 / (1.0f + expf(-g1)) * u1);
    pk[i] = *reinterpret_cast<const uint32_t *>(&b);
  }
  uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v) store16(d + v, make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]));
}

__device__ __forceinline__ void store_plain32(__nv_bfloat16 *dst, const uint32_t (&r)[32]) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
    pk[i] = *reinterpret_cast<const uint32_t *>(&b);
  }
  uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v) store16(d + v, make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]));
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                        const __grid_constant__ CUtensorMap map_b1, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + (((smem_addr(smem_raw) + 1023u) & ~1023u) - smem_addr(smem_raw));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStage);
  uint64_t *empty = full + kStages;
  uint64_t *tfull = empty + kStages;
  uint64_t *tempty = tfull + 2;
  uint64_t *done = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int32_t *offs = reinterpret_cast<int32_t *>(tmem_slot + 2);
  int32_t *pref = offs + (a.E + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 4);
    }
    mbar_init(done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (tid == 32) {
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b0);
    prefetch_tensormap(&map_b1);
  }
  // the offsets and rows come from the previous kernel; tensor memory is only
  // claimed once that kernel has finished
  grid_dependency_wait();
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  for (int e = tid; e <= a.E; e += kGemmThreads) offs[e] = a.region_offsets[static_cast<int64_t>(e) * a.R];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) tile_prefix<kBM>(offs, pref, a, lane);
  __syncthreads();
  const int total = tile_total(pref, a);
  const int kblocks = a.K / kBK;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      uint32_t it = 0;  // K blocks issued
      const uint32_t bytes = kTileA + a.b_rows * kBK * 2;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
        const Tile t = tile_of<kBM>(w, pref, offs, a);
        const int brow = t.e * a.expert_rows + t.n0;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!role_wait(empty + s, ph ^ 1u, abort, a.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_addr(smem + s * kStage), sb = sa + kTileA, fb = smem_addr(full + s);
          mbar_arrive_expect_tx(full + s, bytes);
          tma_load_2d(sa, &map_a, kb * kBK, t.row0, fb);
          if (a.swiglu) {
            tma_load_2d(sb, &map_b0, kb * kBK, brow, fb);
            tma_load_2d(sb + kBoxBytes, &map_b1, kb * kBK, brow, fb);
          } else {
            tma_load_2d(sb, &map_b0, kb * kBK, brow, fb);
            if (a.b_rows > kBoxRows) tma_load_2d(sb + kBoxBytes, &map_b0, kb * kBK, brow + kBoxRows, fb);
          }
          ++it;
        }
      }
      // the last load issued into each stage lands before the CTA may exit
      for (uint32_t s = 0; s < kStages && s < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / kStages) * kStages;
        mbar_wait_bounded(full + s, (last / kStages) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      uint32_t it = 0;
      int lt = 0;
      const uint32_t idesc = idesc_bf16(kBM, a.b_rows);
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++lt) {
        const int buf = lt & 1;
        const uint32_t ph = (lt >> 1) & 1;
        if (!role_wait(tempty + buf, ph ^ 1u, abort, a.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kBNMax;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % kStages, sph = (it / kStages) & 1u;
          if (!role_wait(full + s, sph, abort, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + s * kStage), sb = sa + kTileA;
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk)
            mma_bf16(d, sw128_desc(sa + kk * kUK * 2), sw128_desc(sb + kk * kUK * 2), idesc, (kb | kk) != 0);
          mma_commit(smem_addr(empty + s));
          ++it;
        }
        if (ok) mma_commit(smem_addr(tfull + buf));
      }
      // every MMA issued completes before the tensor memory is freed
      mma_commit(smem_addr(done));
      mbar_wait_bounded(done, 0);
    }
    __syncwarp();
  } else {
    // ---- epilogue: warps 2..5, warp w reads TMEM lanes 32 * (w % 4) .. + 31 ----
    const int q = warp & 3;
    const int m = q * 32 + lane;
    int lt = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++lt) {
      const int buf = lt & 1;
      const uint32_t ph = (lt >> 1) & 1;
      int ok = 0;
      if (lane == 0) ok = role_wait(tfull + buf, ph, abort, a.err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const Tile t = tile_of<kBM>(w, pref, offs, a);
      const bool valid = m < t.rows;
      __nv_bfloat16 *orow = a.out + static_cast<int64_t>(t.row0 + (valid ? m : 0)) * a.n_total + t.n0;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kBNMax;
      if (a.swiglu) {
        for (int c = 0; c < kBNMax / 2; c += 32) {
          uint32_t r[64];
          tmem_load32x2_wait(tb + c, tb + kBNMax / 2 + c, r);
          if (valid) store_swiglu32(orow + c, r);
        }
      } else {
        for (int c = 0; c < a.b_rows; c += 32) {
          uint32_t r[32];
          tmem_load32_wait(tb + c, r);
          if (valid) store_plain32(orow + c, r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(tempty + buf));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (tcgen05 cta_group::2): a cluster of two CTAs on the two
// SMs of a TPC computes a 256 x 256 tile with M = 256 MMAs. CTA r holds rows
// 128 r .. 128 r + 127 of the tile's A rows and half of its B tile (gate rows
// in CTA 0 and up rows in CTA 1 for linear 1; weight rows 0-127 and 128-255
// for linear 2); each CTA's tensor memory receives its 128 rows x 256 columns.
// Each SM reads only its own half of the operands from shared memory, so a K
// block costs 32 KB of shared memory per SM instead of 48 KB.
//   Both CTAs' TMA loads complete on the leader's (rank 0) full barrier, which
//   the leader arms with both halves' bytes; the leader issues the MMAs and
//   commits to the barriers of both CTAs (multicast arrive); each epilogue
//   releases an accumulator by arriving on the leader's tmem-empty barrier.
// ---------------------------------------------------------------------------
#ifndef MOE_GEMM_PAIR_STAGES
#define MOE_GEMM_PAIR_STAGES 6
#endif
constexpr int kPairStages = MOE_GEMM_PAIR_STAGES;
constexpr int kPairStage = kTileA + kBoxBytes;  // this CTA's A rows + its half of B
#ifndef MOE_GEMM_PAIR_TMEM_COLS
#define MOE_GEMM_PAIR_TMEM_COLS 512
#endif
constexpr uint32_t kPairTmemCols = MOE_GEMM_PAIR_TMEM_COLS;
constexpr int kPairBufs = static_cast<int>(kPairTmemCols) / kBNMax;  // accumulators per CTA
constexpr int kPairSmemFixed = 1024 + kPairStages * kPairStage + (2 * kPairStages + 2 * kPairBufs + 1) * 8 + 16;
static_assert(kPairBufs == 1 || kPairBufs == 2, "");
static_assert(kPairStage % 1024 == 0, "");
static_assert(idesc_bf16(256, 256) == 0x10400490u, "");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Shared-memory address of the same location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA tile load into this CTA's shared memory, completing on an mbarrier that may
// live in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at this offset in both CTAs of the pair when every
// tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(both)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Stop both CTAs of the pair: the local flag and the peer's.
__device__ __forceinline__ void abort_pair(volatile int *abort) {
  *abort = 1;
  const uint32_t peer = map_rank(smem_addr(const_cast<int *>(abort)), cluster_rank() ^ 1u);
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer), "r"(1) : "memory");
}

// role_wait with cluster-scope acquire (the barrier is completed from the pair)
// and a pair-wide abort.
__device__ __forceinline__ bool pair_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int32_t *err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kMbarWaitNs) {
      abort_pair(abort);
      latch_error(err, MOE_ETIMEOUT);
      return false;
    }
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                             const __grid_constant__ CUtensorMap map_b1, const GemmArgs a) {
  constexpr int BMP = 2 * kBM;  // rows of a pair tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + (((smem_addr(smem_raw) + 1023u) & ~1023u) - smem_addr(smem_raw));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kPairStages * kPairStage);
  uint64_t *empty = full + kPairStages;
  uint64_t *tfull = empty + kPairStages;
  uint64_t *tempty = tfull + kPairBufs;
  uint64_t *done = tempty + kPairBufs;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *mismatch = reinterpret_cast<volatile int *>(tmem_slot + 2);
  int32_t *offs = reinterpret_cast<int32_t *>(tmem_slot + 4);
  int32_t *pref = offs + (a.E + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  if (tid == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < kPairBufs; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 8);  // four epilogue warps in each CTA
    }
    mbar_init(done, 1);
    *abort = 0;
    *mismatch = 0;
    fence_mbar_init();
  }
  if (tid == 32) {
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b0);
    prefetch_tensormap(&map_b1);
  }
  cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive
  grid_dependency_wait();
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kPairTmemCols);
    tmem_relinquish_pair();
  }
  for (int e = tid; e <= a.E; e += kGemmThreads) offs[e] = a.region_offsets[static_cast<int64_t>(e) * a.R];
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the pair's MMAs address both CTAs' tensor memory at the leader's column:
  // the two allocations must agree
  if (!leader && tid == 0) {
    uint32_t lead;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(lead) : "r"(map_rank(smem_addr(tmem_slot), 0)));
    if (lead != tmem_base) {
      *mismatch = 1;
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(map_rank(smem_addr(const_cast<int *>(mismatch)), 0)),
                   "r"(1)
                   : "memory");
      latch_error(a.err, MOE_ECUDA);
    }
  }
  if (warp == 0) tile_prefix<BMP>(offs, pref, a, lane);
  cluster_sync_all();
  const int total = *mismatch ? 0 : tile_total(pref, a);
  const int kblocks = a.K / kBK;
  const int first = static_cast<int>(cluster_index()), stride = static_cast<int>(cluster_count());

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer (both CTAs): this CTA's rows and half of B ----
      uint32_t it = 0;
      const CUtensorMap *mb = (a.swiglu && !leader) ? &map_b1 : &map_b0;
      bool ok = true;
      for (int w = first; ok && w < total; w += stride) {
        const Tile t = tile_of<BMP>(w, pref, offs, a);
        const int brow = t.e * a.expert_rows + t.n0 + (a.swiglu ? 0 : static_cast<int>(rank) * kBoxRows);
        const int arow = t.row0 + static_cast<int>(rank) * kBM;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % kPairStages, ph = (it / kPairStages) & 1u;
          if (!pair_wait(empty + s, ph ^ 1u, abort, a.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_addr(smem + s * kPairStage), fb = map_rank(smem_addr(full + s), 0);
          if (leader) mbar_arrive_expect_tx(full + s, 2 * kPairStage);
          tma_load_2d_pair(sa, &map_a, kb * kBK, arow, fb);
          tma_load_2d_pair(sa + kTileA, mb, kb * kBK, brow, fb);
          ++it;
        }
      }
      if (leader) {
        // the last loads armed into each stage (both CTAs' halves) land before the pair may exit
        for (uint32_t s = 0; s < kPairStages && s < it; ++s) {
          const uint32_t last = s + ((it - 1 - s) / kPairStages) * kPairStages;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait_cluster(full + s, (last / kPairStages) & 1u) && global_timer_ns() - t0 < kMbarWaitNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---- MMA issuer (leader only) ----
      uint32_t it = 0;
      int lt = 0;
      const uint32_t idesc = idesc_bf16(BMP, kBNMax);
      bool ok = true;
      for (int w = first; ok && w < total; w += stride, ++lt) {
        const int buf = lt % kPairBufs;
        const uint32_t ph = (lt / kPairBufs) & 1;
        if (!pair_wait(tempty + buf, ph ^ 1u, abort, a.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kBNMax;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % kPairStages, sph = (it / kPairStages) & 1u;
          if (!pair_wait(full + s, sph, abort, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + s * kPairStage), sb = sa + kTileA;
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk)
            mma_bf16_pair(d, sw128_desc(sa + kk * kUK * 2), sw128_desc(sb + kk * kUK * 2), idesc, (kb | kk) != 0);
          mma_commit_pair(smem_addr(empty + s));
          ++it;
        }
        if (ok) mma_commit_pair(smem_addr(tfull + buf));
      }
      mma_commit_pair(smem_addr(done));
    }
    __syncwarp();
  } else {
    // ---- epilogue (both CTAs): this CTA's 128 rows of the pair tile ----
    const int q = warp & 3;
    const int m = static_cast<int>(rank) * kBM + q * 32 + lane;  // row within the pair tile
    int lt = 0;
    for (int w = first; w < total; w += stride, ++lt) {
      const int buf = lt % kPairBufs;
      const uint32_t ph = (lt / kPairBufs) & 1;
      int ok = 0;
      if (lane == 0) ok = pair_wait(tfull + buf, ph, abort, a.err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const Tile t = tile_of<BMP>(w, pref, offs, a);
      const bool valid = m < t.rows;
      __nv_bfloat16 *orow = a.out + static_cast<int64_t>(t.row0 + (valid ? m : 0)) * a.n_total + t.n0;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kBNMax;
      if (a.swiglu) {
        for (int c = 0; c < kBNMax / 2; c += 32) {
          uint32_t r[64];
          tmem_load32x2_wait(tb + c, tb + kBNMax / 2 + c, r);
          if (valid) store_swiglu32(orow + c, r);
        }
      } else {
        for (int c = 0; c < kBNMax; c += 32) {
          uint32_t r[32];
          tmem_load32_wait(tb + c, r);
          if (valid) store_plain32(orow + c, r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(map_rank(smem_addr(tempty + buf), 0));
    }
  }
  __syncthreads();
  if (tid == 32) {
    // every MMA of the pair (which reads this CTA's shared memory and writes its
    // tensor memory) has completed
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_cluster(done, 0) && global_timer_ns() - t0 < kMbarWaitNs) {
    }
  }
  if (*abort) {
    // loads this CTA issued towards the leader's barriers may still be landing
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 100000ull) {
    }
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPairTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
int gemm_smem_bytes(int E) { return kSmemFixed + 12 * (E + 1); }  // offsets + two class prefixes
int pair_smem_bytes(int E) { return kPairSmemFixed + 12 * (E + 1); }

// Whether a launch takes the CTA-pair kernel. It needs 256-row B tiles, and it
// pays only for experts with many rows: its 256-row tiles waste half their
// loads and MMAs on an expert of at most 128 rows, where the weights bound the
// kernel anyway. Measured on the Mixtral shape under the GPU's power cap, it
// wins for linear 2 (1.58 against 1.51 PFLOP/s) and loses for linear 1 with
// SwiGLU (1.54 against 1.62: it reads three times the DRAM bytes of the
// single-CTA kernel there), so it is taken for linear 2 only.
// MOE_GEMM_PAIR: 0 never, 1 as above (expected rows per expert R*T*k / E of at
// least kPairMinRows), 2 for every launch with 256-row B tiles (tests).
#ifndef MOE_GEMM_PAIR
#define MOE_GEMM_PAIR 1
#endif
constexpr int kPairMinRows = 512;
bool use_pair(const GemmArgs &a) {
  if (MOE_GEMM_PAIR == 0 || a.b_rows != kBNMax) return false;
  return MOE_GEMM_PAIR == 2 || (!a.swiglu && a.rows / a.E >= kPairMinRows);
}

moe_status launch_pair(const GemmArgs &a, const CUtensorMap &ma, const CUtensorMap &mb0, const CUtensorMap &mb1,
                       int num_sms, cudaStream_t stream) {
  const int smem = pair_smem_bytes(a.E);
  if (smem > kSmemMax) return MOE_EINVAL;
  const int64_t max_tiles = (static_cast<int64_t>(a.rows) / (2 * kBM) + a.E) * a.ntiles_n;
  if (cudaFuncSetAttribute(grouped_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return MOE_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // one persistent cluster per co-resident pair of SMs
  const int sms = num_sms > 0 ? num_sms : sm_count();
  cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, grouped_gemm_pair_kernel, &cfg) != cudaSuccess || active < 1)
    return MOE_ECUDA;
  int64_t clusters = sms / 2 < active ? sms / 2 : active;
  if (clusters > max_tiles) clusters = max_tiles;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  if (cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel, ma, mb0, mb1, a) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

int group_width(const GemmArgs &a, int concurrent, int tile_rows) {
  int64_t g = MOE_GEMM_GROUP_N;
  if (g <= 0) {
    g = std::llround(std::sqrt(static_cast<double>(concurrent) * tile_rows / a.b_rows));
    const int64_t cap = MOE_GEMM_L2_GROUP_BYTES / (static_cast<int64_t>(a.b_rows) * a.K * 2);
    if (g > cap) g = cap;
  }
  return static_cast<int>(g < 1 ? 1 : (g > a.ntiles_n ? a.ntiles_n : g));
}

moe_status launch_grouped(GemmArgs a, const void *A, const void *B0, const void *B1, int64_t b_total_rows,
                          int num_sms, cudaStream_t stream) {
  const int sms_all = num_sms > 0 ? num_sms : sm_count();
  // a CTA pair needs two SMs: with one, the one-CTA kernel runs every launch
  const bool pair = use_pair(a) && sms_all >= 2;
  a.group_n = pair ? group_width(a, sms_all / 2, 2 * kBM) : group_width(a, sms_all, kBM);
  const int smem = gemm_smem_bytes(a.E);
  if (smem > kSmemMax) return MOE_EINVAL;
  const int64_t max_tiles = (static_cast<int64_t>(a.rows) / kBM + a.E) * a.ntiles_n;
  if (max_tiles > INT32_MAX) return MOE_EINVAL;
  CUtensorMap ma, mb0, mb1;
  if (!make_map(&ma, A, a.K, a.rows) || !make_map(&mb0, B0, a.K, b_total_rows) ||
      !make_map(&mb1, B1, a.K, b_total_rows))
    return MOE_ECUDA;
  if (pair) return launch_pair(a, ma, mb0, mb1, num_sms, stream);
  if (cudaFuncSetAttribute(grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return MOE_ECUDA;
  const int sms = num_sms > 0 ? num_sms : sm_count();
  const int64_t grid = max_tiles < sms ? max_tiles : sms;
  if (grid <= 0) return MOE_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  if (cudaLaunchKernelEx(&cfg, grouped_gemm_kernel, ma, mb0, mb1, a) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

// Checks shared by both linear maps; fills rows (= R * T * k packed rows).
moe_status check_expert(const moe_desc *desc, int32_t inter, Sizes *s, int64_t *rows) {
  moe_status st = check_desc(desc, s);
  if (st != MOE_OK) return st;
  if (s->dtype != MOE_BF16) return MOE_EINVAL;
  if (s->H % 128 != 0 || inter < 128 || inter % 128 != 0) return MOE_EINVAL;
  if (static_cast<int64_t>(s->E) * inter > INT32_MAX || static_cast<int64_t>(s->E) * s->H > INT32_MAX)
    return MOE_EINVAL;
  *rows = s->ntok * s->k;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_expert_gate_up(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                         const void *packed_x, const void *w_gate, const void *w_up, void *h,
                                         int32_t *err, void *stream) {
  Sizes s;
  int64_t rows = 0;
  moe_status st = check_expert(desc, inter, &s, &rows);
  if (st != MOE_OK) return st;
  if (region_offsets == nullptr || err == nullptr || !aligned4(region_offsets) || !aligned4(err)) return MOE_EINVAL;
  if (rows == 0) return MOE_OK;
  if (packed_x == nullptr || w_gate == nullptr || w_up == nullptr || h == nullptr) return MOE_EINVAL;
  if (!aligned16(packed_x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(h)) return MOE_EINVAL;
  GemmArgs a{region_offsets, err, static_cast<__nv_bfloat16 *>(h), static_cast<int>(rows), s.E, s.R, s.H,
             inter, kBNMax, kBNMax / 2, inter / (kBNMax / 2), inter, 1, 1};
  return launch_grouped(a, packed_x, w_gate, w_up, static_cast<int64_t>(s.E) * inter, desc->num_sms,
                        static_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_expert_down(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                      const void *h, const void *w_down, void *packed_y, int32_t *err,
                                      void *stream) {
  Sizes s;
  int64_t rows = 0;
  moe_status st = check_expert(desc, inter, &s, &rows);
  if (st != MOE_OK) return st;
  if (region_offsets == nullptr || err == nullptr || !aligned4(region_offsets) || !aligned4(err)) return MOE_EINVAL;
  if (rows == 0) return MOE_OK;
  if (h == nullptr || w_down == nullptr || packed_y == nullptr) return MOE_EINVAL;
  if (!aligned16(h) || !aligned16(w_down) || !aligned16(packed_y)) return MOE_EINVAL;
  const int bn = s.H % kBNMax == 0 ? kBNMax : kBoxRows;
  GemmArgs a{region_offsets, err, static_cast<__nv_bfloat16 *>(packed_y), static_cast<int>(rows), s.E, s.R,
             inter, s.H, bn, bn, s.H / bn, s.H, 0, 1};
  return launch_grouped(a, h, w_down, w_down, static_cast<int64_t>(s.E) * s.H, desc->num_sms,
                        static_cast<cudaStream_t>(stream));
}

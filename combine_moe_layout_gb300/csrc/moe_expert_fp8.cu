// fp8 expert stage: the same two linear maps as moe_expert.cu on e4m3 rows and
// weights with fp32 block scales, on the tensor cores' fp8 path
// (tcgen05.mma.kind::f8f6f4).
//
// "How GPUs Talk to Each Other During LLM Inference", section 7 (Mega MoE):
// every expert applies linear 1, SwiGLU and linear 2 between dispatch and
// combine. "NVSHMEM and DeepEP", high-throughput section: the rows travel as FP8
// with one fp32 scale per 128 elements, which is what the receive hook packs.
// Weights carry one fp32 scale per 128 x 128 block. A value is its e4m3 code
// times its scale, so one 128-wide K block of a dot product is
//   sa[m][kb] * sb[n / 128][kb] * sum_{k in kb} qa[m][k] qb[n][k],
// and the kernel accumulates each K block's code products on the tensor cores
// in fp32 (a "partial" in tensor memory) and then adds it, times the two
// scales, into fp32 registers ("promotion").
//
//   gate/up:  hv = silu(g) * u per row, then per 128 contiguous columns
//             scale = amax / 448 (1 for an all-zero block) and
//             code = e4m3(hv / scale) (RNE, saturating), the dispatch rule,
//             so linear 2 reads e4m3 rows with 128-element scales.
//   down:     y = bf16(sum), round to nearest even.
//
// Kernel shape: one persistent CTA per SM, 384 threads in three warpgroups;
// warpgroup 0 runs with 56 registers a thread and the others with 224
// (setmaxnreg), so the promotion warps keep 128 fp32 sums in registers.
//   warp 0      TMA producer: a 128-row x 128-byte A tile and a 256-row B tile
//               per K block (one scale block), 128-byte swizzle, 3 or 4
//               stages (the kernel's two forms, below).
//   warp 1      owns 512 TMEM columns (two 128 x 256 fp32 partials) and issues
//               4 MMAs (M 128, N 256 or 128, K 32) per K block into one
//               partial, alternating partials so the next K block's MMAs run
//               while the previous partial is promoted. It commits once per K
//               block: the same barrier frees the stage for the producer and
//               hands the partial to the promotion. Warps 2-3 idle.
//   warps 4-11  promotion and epilogue: warp w reads TMEM lanes 32 (w % 4) ..
//               +31 (the tile's rows) and one half of the columns; it adds the
//               scaled partial into 128 fp32 registers and, after the last K
//               block, stores the row's part of the tile: directly, or, in the
//               form for experts of many rows, through its own staging rows in
//               shared memory, so that each store instruction writes whole
//               128-byte lines of 4 rows (64-byte pieces of 8 rows for h) rather
//               than 16 bytes of 32 rows. For gate/up a warp
//               holds gate and up columns of the same 64 intermediate indices,
//               and the two warps that share a row exchange their halves of
//               the block amax through shared memory (an mbarrier, no named
//               barrier, so an aborted partner cannot hang the other).
// Tile order, bounded waits and teardown follow moe_expert.cu.
#include <cuda_bf16.h>

#include <cmath>

#include "moe_tc.cuh"

namespace moe {
namespace {

constexpr int kF8BM = 128;                      // rows of a tile
constexpr int kF8BK = 128;                      // K per stage: one 128-byte row of e4m3, one scale block
constexpr int kF8UK = 32;                       // K of one tcgen05.mma kind::f8f6f4
constexpr int kF8BN = 256;                      // accumulator columns of a tile
constexpr int kF8TileA = kF8BM * kF8BK;         // 16 KB
constexpr int kF8TileB = kF8BN * kF8BK;         // 32 KB
constexpr int kF8Stage = kF8TileA + kF8TileB;
constexpr int kF8BoxBytes = kBoxRows * kF8BK;   // one 128 x 128-byte box
constexpr int kF8PromoWarps = 8;
// Two forms, picked per launch (template parameters STAGES, STAGED):
// - experts with many rows (the tensor cores bound the kernel): 3 stages and a
//   staged epilogue. Each promotion warp writes its 32 rows of up to 128 output
//   bytes per row into its own 4 KB of shared memory and stores them back as
//   whole 128-byte lines (gate/up: 64-byte pieces of h), not one 16-byte piece
//   of 32 different rows per store instruction. With two partials the MMAs run
//   at most one K block ahead of the promotion, and a fourth stage measured no
//   faster there; its shared memory holds the staging rows instead.
// - experts with fewer rows than one tile (the weight stream bounds the kernel):
//   4 stages, for the deeper weight prefetch, and direct stores of the little
//   output there is.
constexpr int kF8OutBytes = 4096;
constexpr int kF8Threads = 128 + 32 * kF8PromoWarps;  // warpgroup 0: TMA, MMA (+2 idle); warpgroups 1-2: promotion
// Register split by warpgroup (setmaxnreg): the block is launched with 168
// registers a thread (384 threads x 168 = 64512); warpgroup 0 gives back to 56
// and the two promotion warpgroups take 224: 128 x 56 + 256 x 224 = 64512.
constexpr int kF8LaunchRegs = 168;
constexpr int kF8CtrlRegs = 56;
constexpr int kF8PromoRegs = 224;
static_assert(128 * kF8CtrlRegs + 256 * kF8PromoRegs <= kF8Threads * kF8LaunchRegs, "register split over budget");
constexpr uint32_t kF8TmemCols = 2 * kF8BN;     // two partials
// stages | epilogue staging (staged form) | full (S), kdone (4), pempty (2), xbar (4), done | slot, abort |
// amax exchange
__host__ __device__ constexpr int f8_smem_fixed(int stages, bool staged) {
  return 1024 + stages * kF8Stage + (staged ? kF8PromoWarps * kF8OutBytes : 0) + (stages + 4 + 2 + 4 + 1) * 8 + 8 +
         2 * 2 * kF8BM * 4;
}
constexpr int kF8SmemMax = 227 * 1024;

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32 (bits 4-5 = 1), A
// and B E4M3 (format 0 in bits 7-9 and 10-12), both K-major, N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
static_assert(idesc_e4m3(128, 256) == 0x08400010u, "");
static_assert(kF8TileA % 1024 == 0 && kF8Stage % 1024 == 0 && kF8BoxBytes % 1024 == 0, "");

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct F8Args {
  const int32_t *region_offsets;  // [E*R + 1]
  int32_t *err;
  const float *a_scales;          // [rows][K/128]
  const float *b_scales;          // [E * expert_rows / 128][K/128]: gate (gate/up) or w_down block scales
  const float *b2_scales;         // up block scales (gate/up); unused for down
  void *out;                      // gate/up: e4m3 [rows][n_total]; down: bf16 [rows][n_total]
  float *out_scales;              // gate/up: [rows][n_total/128]; down: unused
  int rows;
  int E, R;
  int K;                          // contraction length, a multiple of 128
  int n_total;
  int b_rows;                     // weight rows of one B tile: 256 or 128
  int out_cols;                   // output columns of a tile: 128 (gate/up) or b_rows (down)
  int ntiles_n;
  int expert_rows;                // weight rows of one expert (I or H)
  int swiglu;
  int group_n;
};

// TMEM column of promotion chunk c (32 columns) for a warp whose chunks start at
// cbase: gate/up puts chunks 2 and 3 on the up columns, 128 further on.
__device__ __forceinline__ int chunk_col(bool swiglu, int cbase, int c) {
  return swiglu ? (c < 2 ? cbase + 32 * c : 128 + cbase + 32 * (c - 2)) : cbase + 32 * c;
}

template <int N>
__device__ __forceinline__ void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void regs_claim() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// acc[0..1] = f * p[0..1] + acc[0..1], one packed fp32 FMA (each lane rounded as fmaf).
__device__ __forceinline__ void fma2(float f, uint32_t p0, uint32_t p1, float &a0, float &a1) {
  asm("{\n\t.reg .b64 s, x, c, d;\n\t"
      "mov.b64 s, {%2, %2};\n\t"
      "mov.b64 x, {%3, %4};\n\t"
      "mov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 d, s, x, c;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(f), "r"(p0), "r"(p1));
}

// A 2-D TMA tensor store of one box from shared memory, in the CTA's bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <int STAGES, bool STAGED>
__global__ void __launch_bounds__(kF8Threads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                            const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_y,
                            const F8Args a) {
  static_assert(STAGES >= 2 && STAGES <= 4, "the producer's stage wait relies on four kdone barriers");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + (((smem_addr(smem_raw) + 1023u) & ~1023u) - smem_addr(smem_raw));
  uint8_t *ostage = smem + STAGES * kF8Stage;  // [promotion warp][kF8OutBytes], staged form only
  uint64_t *full = reinterpret_cast<uint64_t *>(ostage + (STAGED ? kF8PromoWarps * kF8OutBytes : 0));
  // kdone[i % 4] completes when the MMAs of the CTA's K block i have: it frees
  // stage i % STAGES for the producer and hands partial i % 2 to the promotion
  // (one commit per K block)
  uint64_t *kdone = full + STAGES;
  uint64_t *pempty = kdone + 4;
  uint64_t *xbar = pempty + 2;
  uint64_t *done = xbar + 4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *xamax = reinterpret_cast<float *>(tmem_slot + 2);  // [tile parity][column half][row]
  int32_t *offs = reinterpret_cast<int32_t *>(xamax + 2 * 2 * kF8BM);
  int32_t *pref = offs + (a.E + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(full + s, 1);
    for (int b = 0; b < 4; ++b) mbar_init(kdone + b, 1);
    for (int b = 0; b < 2; ++b) mbar_init(pempty + b, kF8PromoWarps);
    for (int q = 0; q < 4; ++q) mbar_init(xbar + q, 64);  // every lane of the two warps of a row quarter
    mbar_init(done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (tid == 32) {
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b0);
    prefetch_tensormap(&map_b1);
  }
  grid_dependency_wait();
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kF8TmemCols);
    tmem_relinquish();
  }
  for (int e = tid; e <= a.E; e += kF8Threads) offs[e] = a.region_offsets[static_cast<int64_t>(e) * a.R];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (warp == 0) tile_prefix<kF8BM>(offs, pref, a, lane);
  __syncthreads();
  const int total = tile_total(pref, a);
  const int kblocks = a.K / kF8BK;

  if (warp == 0) {
    regs_release<kF8CtrlRegs>();
    if (lane == 0) {
      // ---- TMA producer ----
      uint32_t it = 0;
      const uint32_t bytes = kF8TileA + a.b_rows * kF8BK;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
        const Tile t = tile_of<kF8BM>(w, pref, offs, a);
        const int brow = t.e * a.expert_rows + t.n0;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % STAGES;
          // the stage is free once the MMAs of K block it - STAGES have completed
          // (STAGES <= 4: that barrier cannot have moved on to K block it yet)
          if (it >= STAGES && !role_wait(kdone + ((it - STAGES) & 3u), ((it - STAGES) >> 2) & 1u, abort, a.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_addr(smem + s * kF8Stage), sb = sa + kF8TileA, fb = smem_addr(full + s);
          mbar_arrive_expect_tx(full + s, bytes);
          tma_load_2d(sa, &map_a, kb * kF8BK, t.row0, fb);
          if (a.swiglu) {
            tma_load_2d(sb, &map_b0, kb * kF8BK, brow, fb);
            tma_load_2d(sb + kF8BoxBytes, &map_b1, kb * kF8BK, brow, fb);
          } else {
            tma_load_2d(sb, &map_b0, kb * kF8BK, brow, fb);
            if (a.b_rows > kBoxRows) tma_load_2d(sb + kF8BoxBytes, &map_b0, kb * kF8BK, brow + kBoxRows, fb);
          }
          ++it;
        }
      }
      for (uint32_t s = 0; s < STAGES && s < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / STAGES) * STAGES;
        mbar_wait_bounded(full + s, (last / STAGES) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    regs_release<kF8CtrlRegs>();
    if (lane == 0) {
      // ---- MMA issuer: one partial per K block, two partials alternating ----
      uint32_t it = 0, pk = 0;
      const uint32_t idesc = idesc_e4m3(kF8BM, a.b_rows);
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % STAGES, sph = (it / STAGES) & 1u;
          const uint32_t pb = pk & 1u, pph = (pk >> 1) & 1u;
          if (!role_wait(full + s, sph, abort, a.err) || !role_wait(pempty + pb, pph ^ 1u, abort, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + s * kF8Stage), sb = sa + kF8TileA;
          const uint32_t d = tmem_base + pb * kF8BN;
          // K step kk starts kk * 32 bytes further along the swizzled rows: the
          // descriptor's address field (bits 0-13, address >> 4) grows by 2 per step
          const uint64_t da = sw128_desc(sa), db = sw128_desc(sb);
#pragma unroll
          for (int kk = 0; kk < kF8BK / kF8UK; ++kk)
            mma_e4m3(d, da + static_cast<uint64_t>(kk * kF8UK / 16), db + static_cast<uint64_t>(kk * kF8UK / 16), idesc,
                     kk != 0);
          mma_commit(smem_addr(kdone + (it & 3u)));
          ++it;
          ++pk;
        }
      }
      mma_commit(smem_addr(done));
      mbar_wait_bounded(done, 0);
    }
    __syncwarp();
  } else if (warp < 4) {
    regs_release<kF8CtrlRegs>();  // warps 2-3: idle
  } else {
    regs_claim<kF8PromoRegs>();
    // ---- promotion and epilogue: warps 4..11 ----
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int j = (warp - 4) >> 2;       // column half
    const int m = q * 32 + lane;         // row within the tile
    const int k128 = a.K / kF8BK;
    // the 32-column chunks this warp promotes: gate/up takes gate columns
    // 64j..64j+63 and the up columns 128 apart (chunks 2, 3 take the up scale);
    // down takes 128 (or, for 128-wide tiles, 64) contiguous columns of half j
    const int ncol = (a.swiglu || a.b_rows == kF8BN) ? 4 : 2;
    const int cbase = a.swiglu ? 64 * j : (a.b_rows == kF8BN ? 128 * j : 64 * j);
    const bool sw = a.swiglu != 0;
    uint32_t pk = 0;
    int lt = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++lt) {
      const Tile t = tile_of<kF8BM>(w, pref, offs, a);
      const bool valid = m < t.rows;
      const int64_t arow = valid ? t.row0 + m : t.row0;
      // weight block rows of this warp's scales
      const int64_t blk = (static_cast<int64_t>(t.e) * a.expert_rows + t.n0 +
                           ((!a.swiglu && a.b_rows == kF8BN) ? 128 * j : 0)) / 128;
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      bool ok = true;
      // the K block's scales, loaded one K block ahead
      const float *sa_p = a.a_scales + arow * k128, *sb_p = a.b_scales + blk * k128;
      const float *sb2_p = a.b2_scales + blk * k128;
      float sa_n = __ldg(sa_p), sb_n = __ldg(sb_p), sb2_n = sw ? __ldg(sb2_p) : 0.0f;
      for (int kb = 0; kb < kblocks; ++kb, ++pk) {
        const float sa = sa_n, sb = sb_n, sb2 = sb2_n;
        if (kb + 1 < kblocks) {
          sa_n = __ldg(sa_p + kb + 1);
          sb_n = __ldg(sb_p + kb + 1);
          if (sw) sb2_n = __ldg(sb2_p + kb + 1);
        }
        const float f0 = sa * sb;
        const float f1 = sw ? sa * sb2 : f0;
        const uint32_t pb = pk & 1u;
        // every lane polls the barrier (measured 2-3% faster than one lane and a
        // broadcast); the vote keeps the warp together if a bounded wait gives up
        const bool got = __all_sync(0xffffffffu, role_wait(kdone + (pk & 3u), (pk >> 2) & 1u, abort, a.err));
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + pb * kF8BN;
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
          if (c < ncol) {
            uint32_t r[64];
            tmem_load32x2_wait(tb + chunk_col(sw, cbase, c), tb + chunk_col(sw, cbase, c + 1), r);
            if (c + 2 >= ncol) {
              // the partial has been read: the MMA warp may refill it
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_local(pempty + pb);
            }
            const float f = (sw && c >= 2) ? f1 : f0;
#pragma unroll
            for (int i = 0; i < 64; i += 2) fma2(f, r[i], r[i + 1], acc[32 * c + i], acc[32 * c + i + 1]);
          }
        }
      }
      if (!ok) break;
      if (a.swiglu) {
        // hv = silu(g) * u for this warp's 64 intermediate indices, in place, with
        // the fast exponential and division (a few ulps, far inside the fp32
        // accumulation error of g and u): the promotion warps run this epilogue
        // while the MMAs wait for their partials, and the IEEE forms made linear 1
        // 7% slower on the DeepSeek prefill shape (7.49 against 6.94 ms)
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float g = acc[i];
          acc[i] = __fdividef(g, 1.0f + __expf(-g)) * acc[64 + i];
          part = fmaxf(part, fabsf(acc[i]));
        }
        // the 128-column block amax: this warp's half and its partner's
        float *slot = xamax + (lt & 1) * 2 * kF8BM;
        slot[j * kF8BM + m] = part;
        mbar_arrive_local(xbar + q);
        if (!__all_sync(0xffffffffu, role_wait(xbar + q, static_cast<uint32_t>(lt & 1), abort, a.err))) break;
        const float amax = fmaxf(part, slot[(j ^ 1) * kF8BM + m]);
        const BlockScale bs = block_scale(amax);
        const float sc = bs.s;
        if constexpr (STAGED) {
          // this lane's 64 codes into its staging row (64 bytes: four 16-byte pieces,
          // piece p at p ^ ((row >> 1) & 3), so that eight rows fill all 32 banks)
          uint4 *buf = reinterpret_cast<uint4 *>(ostage + (warp - 4) * kF8OutBytes);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t pk4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int x = 16 * v + 4 * i;
              const uint16_t lo = e4m3x2_of_quotients(acc[x], acc[x + 1], bs);
              const uint16_t hi = e4m3x2_of_quotients(acc[x + 2], acc[x + 3], bs);
              pk4[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            buf[lane * 4 + (v ^ ((lane >> 1) & 3))] = make_uint4(pk4[0], pk4[1], pk4[2], pk4[3]);
          }
          if (valid && j == 0) a.out_scales[arow * (a.n_total / 128) + t.n0 / 128] = sc;
          __syncwarp();
          // stores of 8 rows x 64 bytes: lane l takes piece l % 4 of row l / 4 + 8 i
          uint8_t *obase = static_cast<uint8_t *>(a.out) + t.n0 + 64 * j;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = (lane >> 2) + 8 * i, pc = lane & 3;
            const uint4 v = buf[r * 4 + (pc ^ ((r >> 1) & 3))];
            if (q * 32 + r < t.rows)
              reinterpret_cast<uint4 *>(obase + static_cast<int64_t>(t.row0 + q * 32 + r) * a.n_total)[pc] = v;
          }
          __syncwarp();
        } else {
          if (valid) {
            uint32_t pk4[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint16_t lo = e4m3x2_of_quotients(acc[4 * i], acc[4 * i + 1], bs);
              const uint16_t hi = e4m3x2_of_quotients(acc[4 * i + 2], acc[4 * i + 3], bs);
              pk4[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            uint8_t *orow = static_cast<uint8_t *>(a.out) + arow * a.n_total + t.n0 + 64 * j;
            uint4 *d = reinterpret_cast<uint4 *>(orow);
#pragma unroll
            for (int v = 0; v < 4; ++v) d[v] = make_uint4(pk4[4 * v], pk4[4 * v + 1], pk4[4 * v + 2], pk4[4 * v + 3]);
            if (j == 0) a.out_scales[arow * (a.n_total / 128) + t.n0 / 128] = sc;
          }
        }
      } else if constexpr (STAGED) {
        // bf16 y, 64 columns at a time: this lane's 128 bytes into its staging row
        // (piece p at p ^ (row & 7): the layout of a TMA box with the 128-byte
        // swizzle). A warp whose 32 rows all belong to the tile stores them with
        // one TMA tensor store and goes on; otherwise the lanes store 4 rows x 128
        // bytes at a time, whole lines: lane l takes piece l % 8 of row l / 8 + 4 i
        uint4 *buf = reinterpret_cast<uint4 *>(ostage + (warp - 4) * kF8OutBytes);
        __nv_bfloat16 *obase = static_cast<__nv_bfloat16 *>(a.out) + t.n0 + cbase;
        const bool whole = q * 32 + 31 < t.rows;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          if (2 * h2 < ncol) {
            // the staging rows are free once the last tensor store has read them
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              uint32_t pk2[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int x = 64 * h2 + 8 * p + 2 * i;
                const __nv_bfloat162 b = __floats2bfloat162_rn(acc[x], acc[x + 1]);
                pk2[i] = *reinterpret_cast<const uint32_t *>(&b);
              }
              buf[lane * 8 + (p ^ (lane & 7))] = make_uint4(pk2[0], pk2[1], pk2[2], pk2[3]);
            }
            if (whole) {
              fence_proxy_async_smem();  // the rows written above, before the async proxy reads them
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&map_y, smem_addr(buf), t.n0 + cbase + 64 * h2, t.row0 + q * 32);
                bulk_commit();
              }
            } else {
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int r = (lane >> 3) + 4 * i, p = lane & 7;
                const uint4 v = buf[r * 8 + (p ^ (r & 7))];
                if (q * 32 + r < t.rows)
                  reinterpret_cast<uint4 *>(obase + static_cast<int64_t>(t.row0 + q * 32 + r) * a.n_total + 64 * h2)[p] =
                      v;
              }
            }
            __syncwarp();
          }
        }
      } else {
        if (valid) {
          __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.out) + arow * a.n_total + t.n0 + cbase;
          uint4 *d = reinterpret_cast<uint4 *>(orow);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (c < ncol) {
              uint32_t pk2[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(acc[32 * c + 2 * i], acc[32 * c + 2 * i + 1]);
                pk2[i] = *reinterpret_cast<const uint32_t *>(&b);
              }
#pragma unroll
              for (int v = 0; v < 4; ++v)
                d[4 * c + v] = make_uint4(pk2[4 * v], pk2[4 * v + 1], pk2[4 * v + 2], pk2[4 * v + 3]);
            }
          }
        }
      }
    }
    // the tensor stores issued from this warp's staging rows have completed
    if constexpr (STAGED) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kF8TmemCols);
  }
}

// 2-D map of the bf16 [rows][cols] output: boxes of 32 rows x 64 columns (128 bytes), 128-byte swizzle.
bool make_map_y(CUtensorMap *map, const void *base, int64_t cols, int64_t rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int fp8_group_width(const F8Args &a, int concurrent) {
  int64_t g = std::llround(std::sqrt(static_cast<double>(concurrent) * kF8BM / a.b_rows));
  const int64_t cap = (64ll << 20) / (static_cast<int64_t>(a.b_rows) * a.K);
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : (g > a.ntiles_n ? a.ntiles_n : g));
}

template <int STAGES, bool STAGED>
moe_status launch_form(const F8Args &a, const CUtensorMap &ma, const CUtensorMap &mb0, const CUtensorMap &mb1,
                       const CUtensorMap &my, int64_t grid, cudaStream_t stream) {
  auto kernel = grouped_gemm_fp8_kernel<STAGES, STAGED>;
  const int smem = f8_smem_fixed(STAGES, STAGED) + 12 * (a.E + 1);  // offsets + two class prefixes
  if (smem > kF8SmemMax) return MOE_EINVAL;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return MOE_ECUDA;
  // the register split needs the launch allocation it was sized for
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess || fa.numRegs < kF8LaunchRegs) return MOE_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kF8Threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  if (cudaLaunchKernelEx(&cfg, kernel, ma, mb0, mb1, my, a) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

moe_status launch_fp8(F8Args a, const void *A, const void *B0, const void *B1, int64_t b_total_rows, int num_sms,
                      cudaStream_t stream) {
  // the larger of the two forms' shared memory decides which expert counts are accepted
  if (f8_smem_fixed(4, false) + 12 * (a.E + 1) > kF8SmemMax || f8_smem_fixed(3, true) + 12 * (a.E + 1) > kF8SmemMax)
    return MOE_EINVAL;
  const int64_t max_tiles = (static_cast<int64_t>(a.rows) / kF8BM + a.E) * a.ntiles_n;
  if (max_tiles > INT32_MAX) return MOE_EINVAL;
  const int sms = num_sms > 0 ? num_sms : sm_count();
  a.group_n = fp8_group_width(a, sms);
  CUtensorMap ma, mb0, mb1, my;
  if (!make_map(&ma, A, a.K, a.rows, 1) || !make_map(&mb0, B0, a.K, b_total_rows, 1) ||
      !make_map(&mb1, B1, a.K, b_total_rows, 1))
    return MOE_ECUDA;
  // linear 2's bf16 output [rows][n_total]: boxes of 32 rows x 64 columns with the 128-byte swizzle, the
  // layout of a promotion warp's staging rows (gate/up writes h with plain stores and never uses the map)
  if (a.swiglu)
    my = ma;
  else if (!make_map_y(&my, a.out, a.n_total, a.rows))
    return MOE_ECUDA;
  const int64_t grid = max_tiles < sms ? max_tiles : sms;
  if (grid <= 0) return MOE_OK;
  // fewer expected rows per expert than one tile: the weight stream bounds the launch
  if (a.rows / a.E < kF8BM) return launch_form<4, false>(a, ma, mb0, mb1, my, grid, stream);
  return launch_form<3, true>(a, ma, mb0, mb1, my, grid, stream);
}

moe_status check_fp8(const moe_desc *desc, int32_t inter, Sizes *s, int64_t *rows) {
  moe_status st = check_desc(desc, s);
  if (st != MOE_OK) return st;
  if (s->dtype == MOE_BF16) return MOE_EINVAL;  // the packed rows must be e4m3 with 128-element scales
  if (s->H % 128 != 0 || inter < 128 || inter % 128 != 0) return MOE_EINVAL;
  if (static_cast<int64_t>(s->E) * inter > INT32_MAX || static_cast<int64_t>(s->E) * s->H > INT32_MAX)
    return MOE_EINVAL;
  *rows = s->ntok * s->k;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_expert_gate_up_fp8(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                             const void *packed_x, const float *packed_scales, const void *w_gate,
                                             const float *w_gate_scales, const void *w_up, const float *w_up_scales,
                                             void *h, float *h_scales, int32_t *err, void *stream) {
  Sizes s;
  int64_t rows = 0;
  moe_status st = check_fp8(desc, inter, &s, &rows);
  if (st != MOE_OK) return st;
  if (region_offsets == nullptr || err == nullptr || !aligned4(region_offsets) || !aligned4(err)) return MOE_EINVAL;
  if (rows == 0) return MOE_OK;
  if (packed_x == nullptr || packed_scales == nullptr || w_gate == nullptr || w_gate_scales == nullptr ||
      w_up == nullptr || w_up_scales == nullptr || h == nullptr || h_scales == nullptr)
    return MOE_EINVAL;
  if (!aligned16(packed_x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(h) || !aligned4(packed_scales) ||
      !aligned4(w_gate_scales) || !aligned4(w_up_scales) || !aligned4(h_scales))
    return MOE_EINVAL;
  F8Args a{region_offsets, err, packed_scales, w_gate_scales, w_up_scales, h, h_scales, static_cast<int>(rows),
           s.E, s.R, s.H, inter, kF8BN, kF8BN / 2, inter / (kF8BN / 2), inter, 1, 1};
  return launch_fp8(a, packed_x, w_gate, w_up, static_cast<int64_t>(s.E) * inter, desc->num_sms,
                    static_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_expert_down_fp8(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                          const void *h, const float *h_scales, const void *w_down,
                                          const float *w_down_scales, void *packed_y, int32_t *err, void *stream) {
  Sizes s;
  int64_t rows = 0;
  moe_status st = check_fp8(desc, inter, &s, &rows);
  if (st != MOE_OK) return st;
  if (region_offsets == nullptr || err == nullptr || !aligned4(region_offsets) || !aligned4(err)) return MOE_EINVAL;
  if (rows == 0) return MOE_OK;
  if (h == nullptr || h_scales == nullptr || w_down == nullptr || w_down_scales == nullptr || packed_y == nullptr)
    return MOE_EINVAL;
  if (!aligned16(h) || !aligned16(w_down) || !aligned16(packed_y) || !aligned4(h_scales) || !aligned4(w_down_scales))
    return MOE_EINVAL;
  const int bn = s.H % kF8BN == 0 ? kF8BN : kBoxRows;
  F8Args a{region_offsets, err, h_scales, w_down_scales, w_down_scales, packed_y, nullptr, static_cast<int>(rows),
           s.E, s.R, inter, s.H, bn, bn, s.H / bn, s.H, 0, 1};
  return launch_fp8(a, h, w_down, w_down, static_cast<int64_t>(s.E) * s.H, desc->num_sms,
                    static_cast<cudaStream_t>(stream));
}

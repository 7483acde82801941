// Tensor-core building blocks shared by the expert-stage GEMM kernels: the
// tcgen05 shared-memory and instruction descriptors, TMA tensor loads,
// tensor-memory allocation, MMA issue and commit, accumulator loads, bounded
// role waits, the expert-by-expert tile order, and the host-side tensor maps.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kBoxRows = 128;  // rows of one TMA box

// tcgen05 shared-memory matrix descriptor of a K-major bf16 tile as TMA writes
// it with the 128-byte swizzle: 128-byte rows (64 elements), 8-row groups 1024
// bytes apart. Fields: start address >> 4 (bits 0-13); leading-dimension byte
// offset >> 4 (bits 16-29; unused by swizzled K-major layouts, 1 by
// convention); stride-dimension byte offset >> 4 (bits 32-45); descriptor
// version 1 (bits 46-48); base offset 0 (bits 49-51: tiles start on 1024-byte
// boundaries); swizzle mode 2 = 128 bytes (bits 61-63).
__host__ __device__ constexpr uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(16 >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, bits 10-12 = 1), no negation, both K-major (bits 15 and
// 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

static_assert(sw128_desc(0x400) == ((2ull << 61) | (1ull << 46) | (64ull << 32) | (1ull << 16) | 0x40ull), "");
static_assert(sw128_desc(0x3FC00 + 96) == ((2ull << 61) | (1ull << 46) | (64ull << 32) | (1ull << 16) | 0x3FC6ull), "");
static_assert(idesc_bf16(128, 256) == 0x08400490u, "");
static_assert(idesc_bf16(128, 128) == 0x08200490u, "");

// ---------------------------------------------------------------------------
// TMA tensor loads, tensor memory and tcgen05.mma.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tmem) = A * B^T (+ D when accumulate != 0), both operands K-major in shared memory.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// tcgen05.ld of 32 consecutive fp32 columns of this thread's accumulator row
// (32x32b shape: lane l of the warp reads TMEM lane base + l), then the wait;
// the wait sits in the same asm block so no use of r can move above it.
__device__ __forceinline__ void tmem_load32_wait(uint32_t taddr0, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr0)
      : "memory");
}

__device__ __forceinline__ void tmem_load32x2_wait(uint32_t taddr0, uint32_t taddr1, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr0), "r"(taddr1)
      : "memory");
}

// Bounded wait on an mbarrier phase that also gives up as soon as another role
// of the CTA has aborted; a timeout records MOE_ETIMEOUT and aborts the CTA.
__device__ __forceinline__ bool role_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int32_t *err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kMbarWaitNs) {
      *abort = 1;
      latch_error(err, MOE_ETIMEOUT);
      return false;
    }
  }
}

struct Tile {
  int e, row0, rows, n0;
};

// The tile sequence. An expert with two or more m-tiles ("hot": its weight
// tiles are read again from L2 by its later m-tiles) has tiles that lean on the
// tensor cores; an expert with one m-tile ("cold") streams its weights once and
// leans on HBM. Each class keeps its own tile prefix, pref[0..E] (hot) and
// pref[E+1..2E+1] (cold), in expert order, and the sequence alternates a hot
// and a cold tile for as long as both last, then runs the rest of the longer
// class. The CTAs running at one time then keep both the tensor cores and HBM
// busy under skewed routing; with one class empty the order is expert order.
template <class Args>
__device__ __forceinline__ int tile_total(const int32_t *pref, const Args &a) {
  return pref[a.E] + pref[2 * a.E + 1];
}

// Tile w of the sequence: its class and index in the class, its expert (the
// class prefix brackets the index), its group of group_n n-tiles (the last
// group may be narrower), then m-tile and, innermost, the n-tile within the
// group.
template <int BM, class Args>
__device__ __forceinline__ Tile tile_of(int w, const int32_t *pref, const int32_t *offs, const Args &a) {
  const int th = pref[a.E], tc = pref[2 * a.E + 1];
  const int both = th < tc ? th : tc;
  int cls, idx;
  if (w < 2 * both) {
    cls = w & 1;
    idx = w >> 1;
  } else {
    cls = th > tc ? 0 : 1;
    idx = both + (w - 2 * both);
  }
  const int32_t *pc = pref + cls * (a.E + 1);
  int lo = 0, hi = a.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pc[mid] <= idx)
      lo = mid;
    else
      hi = mid - 1;
  }
  Tile t;
  t.e = lo;
  const int m = offs[lo + 1] - offs[lo];
  const int mtiles = (m + BM - 1) / BM;
  const int local = idx - pc[lo];
  const int per_group = mtiles * a.group_n;
  const int g = local / per_group, r = local - g * per_group;
  const int gw = min(a.group_n, a.ntiles_n - g * a.group_n);
  const int mt = r / gw, nt = g * a.group_n + (r - mt * gw);
  t.row0 = offs[lo] + mt * BM;
  t.rows = min(BM, m - mt * BM);
  t.n0 = nt * a.out_cols;
  return t;
}

// Tiles per expert and the two class prefixes (one warp); an expert whose rows
// are not a valid range of the packed buffer gets none and latches MOE_EINVAL.
template <int BM, class Args>
__device__ __forceinline__ void tile_prefix(const int32_t *offs, int32_t *pref, const Args &a, int lane) {
  int run_h = 0, run_c = 0;
  bool bad = false;
  for (int e0 = 0; e0 < a.E; e0 += 32) {
    const int e = e0 + lane;
    int hot = 0, cold = 0;
    if (e < a.E) {
      const int lo = offs[e], hi = offs[e + 1];
      if (lo < 0 || hi < lo || hi > a.rows) {
        bad = true;
      } else {
        const int mtiles = (hi - lo + BM - 1) / BM;
        (mtiles >= 2 ? hot : cold) = mtiles * a.ntiles_n;
      }
    }
    int ih = hot, ic = cold;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vh = __shfl_up_sync(0xffffffffu, ih, o);
      const int vc = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) {
        ih += vh;
        ic += vc;
      }
    }
    if (e < a.E) {
      pref[e] = run_h + ih - hot;
      pref[a.E + 1 + e] = run_c + ic - cold;
    }
    run_h += __shfl_sync(0xffffffffu, ih, 31);
    run_c += __shfl_sync(0xffffffffu, ic, 31);
  }
  if (lane == 0) {
    pref[a.E] = run_h;
    pref[2 * a.E + 1] = run_c;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) latch_error(a.err, MOE_EINVAL);
}

// ---------------------------------------------------------------------------
// Host side: tensor maps.
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D map of a row-major [rows][K] matrix of 2-byte (bf16) or 1-byte (e4m3)
// elements, boxes of 128 rows x one 128-byte swizzle row, 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, int64_t K, int64_t rows, int elem_bytes = 2) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * elem_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(kBoxRows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace moe

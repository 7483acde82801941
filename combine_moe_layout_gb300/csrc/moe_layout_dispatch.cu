// Layout and dispatch in one kernel, for decode-sized batches (T <= 1024 tokens
// per rank, rows of at most 16 KiB).
//
// Same results as moe_layout followed by moe_dispatch (Perplexity,
// "Efficient and portable mixture-of-experts communication", section
// "Dispatch": one warp counts the tokens per destination expert while the
// other warps pack the tokens; "NVSHMEM and DeepEP: GPU-initiated
// communication", low-latency section: fixed slots, no exchange). Every CTA is
// such a sender for one row (src, t) at a time:
//   1. all threads load the row into registers (16- or 32-byte vectors), its
//      scales and the row's k experts;
//   2. the CTA reads the routing entries of rank src's earlier tokens
//      (L2-resident after the first CTA) and, per thread, counts the entries
//      equal to each of the row's k experts; warp reductions and one exchange
//      in shared memory give pos_j = entries of tokens t' < t that chose e_j,
//      i.e. the token-order position, with no grid-wide step and no wait on
//      another CTA;
//   3. the last 32 rows of a rank read all of its entries and also histogram
//      a share of the experts, so every (expert, source) count and its
//      count + 1 flag is written by exactly one CTA;
//   4. every thread stores its vectors into the k slots (bf16 rows quantised
//      to e4m3 on the way, for MOE_BF16_TO_FP8); only then are tok_slot, the
//      slot headers, counts and flags written, so a CTA's copies never queue
//      behind them.
// Nothing is read before griddepcontrol.wait, so every input may come from
// the kernel immediately before this one in the stream.
#include <climits>

#include "moe_common.cuh"

namespace moe {

constexpr int kFusedThreads = 128;
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedMaxTokens = 1024;
constexpr int kFusedMaxVec16 = 8;  // 16-byte vectors per thread: rows of at most 128 * 8 * 16 B = 16 KiB
constexpr int kFusedMaxVec32 = 4;  // 32-byte vectors per thread: the same 16 KiB
constexpr int64_t kFusedNarrowMaxRow = 8192;  // plain copies of rows up to this many bytes use 16-byte vectors
constexpr int kFusedMaxHist = 2048;       // experts one CTA histograms (G = ceil(E / T))
constexpr int kFusedScanRegs = 2;        // int4 routing loads per thread issued with the row's loads
constexpr int kFusedHistRows = 32;       // rows per rank that also count experts for counts and flags

struct FusedArgs {
  const int32_t *topk_idx;
  int32_t *counts;
  int32_t *tok_slot;
  const uint8_t *x;
  const float *x_scales;
  SlotParts parts;  // rows, scales, headers and count + 1 flags of the receive side
  int32_t *err;
  int R, T, E, k, max_m, nsc, G, early;
  int vin;      // W-byte vectors of a caller's input row
  int idx_vec;  // a rank's routing can be read as int4 (T*k % 4 == 0, 16-byte aligned base)
  int sc_vec;   // scales move as float4 (nsc % 4 == 0, both scale arrays 16-byte aligned)
  uint32_t row_bytes;     // a dispatched row: the slot stride of the receive rows
  uint32_t in_row_bytes;  // a caller's input row
  int64_t nrows;
};

// A W-byte piece of a row (W = 16 or 32), moved with one vector load and one
// vector store per slot.
template <int W>
struct RowVec {
  uint32_t w[W / 4];
};

// Read-once load (evict-first) of a row piece; volatile keeps it ahead of the
// CTA barriers that follow, so its latency overlaps the layout work.
template <int W>
__device__ __forceinline__ RowVec<W> ld_row(const uint8_t *p) {
  RowVec<W> r;
  if constexpr (W == 32) {
    asm volatile("ld.global.cs.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
                   "=r"(r.w[6]), "=r"(r.w[7])
                 : "l"(p));
  } else {
    asm volatile("ld.global.cs.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "l"(p));
  }
  return r;
}

// L2 policy of the slot rows: evict last. The experts read the slots next, and
// the combine that follows a step reads 117 MB (decode) through L2: measured on
// GB300, with the 60 MB of slot rows held at normal priority that combine took
// 26.4 us, with evict-last 24.7 us, the same as after a clean L2.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

template <int W>
__device__ __forceinline__ void st_row(uint8_t *p, const RowVec<W> &r, uint64_t pol) {
  if constexpr (W == 32) {
    asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p),
                 "r"(r.w[0]), "r"(r.w[1]), "r"(r.w[2]), "r"(r.w[3]), "r"(r.w[4]), "r"(r.w[5]), "r"(r.w[6]),
                 "r"(r.w[7]), "l"(pol)
                 : "memory");
  } else {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(r.w[0]), "r"(r.w[1]),
                 "r"(r.w[2]), "r"(r.w[3]), "l"(pol)
                 : "memory");
  }
}

// The quantising forms would take up to 96 registers a thread, 5 CTAs per SM:
// 760 of a decode batch's 1024 rows at a time, then a second wave. Capped at 72
// (7 CTAs per SM, every row of the batch at once, a few words spilled), the
// 1024-row bf16 decode batch measured 20.3 against 24.3 us. The other forms
// give 0, which leaves the register count to the compiler as with no bound (an
// explicit 1 let it grow the fp8 decode form from 62 to 100 registers, 4 CTAs
// per SM, and that step from 36.8 to 38.3 us).
template <int W, int VPT, int KC, bool QUANT>
__global__ void __launch_bounds__(kFusedThreads, QUANT ? 7 : 0) layout_dispatch_kernel(FusedArgs a) {
  __shared__ int32_t s_part[kFusedWarps][KC];
  __shared__ int32_t s_own[KC];
  __shared__ int32_t s_slot[KC];
  __shared__ uint8_t *s_dst[KC];  // each choice's slot row (in its part)
  __shared__ float *s_dsc[KC];    // and its scales
  extern __shared__ int32_t s_hist[];  // [G]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // every input (x, x_scales, topk_idx) may be written by the previous kernel
  grid_dependency_wait();
  if (a.early) grid_dependents_launch();

  const int n = a.T * a.k;  // routing entries of a rank
  const int hist_rows = min(a.T, kFusedHistRows);
  for (int64_t row = blockIdx.x; row < a.nrows; row += gridDim.x) {
    const int src = static_cast<int>(row / a.T);
    const int t = static_cast<int>(row - static_cast<int64_t>(src) * a.T);
    const int32_t *ridx = a.topk_idx + static_cast<int64_t>(src) * a.T * a.k;  // routing of rank src
    const int32_t *own_p = ridx + static_cast<int64_t>(t) * a.k;

    // 1. every load of the row at once: the row, its scales, its experts and
    //    the first kFusedScanRegs entries per thread of the rank's routing
    RowVec<W> v[VPT];
    const uint8_t *xr = a.x + row * a.in_row_bytes;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      const int q = tid + u * kFusedThreads;
      if (q < a.vin) {
        v[u] = ld_row<W>(xr + static_cast<int64_t>(q) * W);
      } else {
#pragma unroll
        for (int z = 0; z < W / 4; ++z) v[u].w[z] = 0;
      }
    }
    float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!QUANT && a.nsc > 0) {
      const float *xs = a.x_scales + row * a.nsc;
      if (a.sc_vec) {
        if (tid < a.nsc / 4) sc = __ldcs(reinterpret_cast<const float4 *>(xs) + tid);
      } else if (tid < a.nsc) {
        sc.x = __ldcs(xs + tid);
      }
    }
    // The last hist_rows rows of a rank also count experts [h0, h0 + hn) over
    // all of its entries (they visit nearly all of them anyway); the other rows
    // visit only the entries of earlier tokens.
    const int hr = t - (a.T - hist_rows);
    const int h0 = hr >= 0 ? hr * a.G : 0;
    const int hn = hr >= 0 ? max(0, min(a.G, a.E - h0)) : 0;
    const int before = t * a.k;
    const int m = hn > 0 ? n : before;  // entries this CTA visits
    int4 r4[kFusedScanRegs];
    if (a.idx_vec) {
#pragma unroll
      for (int c = 0; c < kFusedScanRegs; ++c) {
        const int q = tid + c * kFusedThreads;
        r4[c] = 4 * q < m ? __ldcg(reinterpret_cast<const int4 *>(ridx) + q) : make_int4(-1, -1, -1, -1);
      }
    }
    if (tid < a.k) {
      const int e = __ldcg(own_p + tid);
      s_own[tid] = (e >= 0 && e < a.E) ? e : INT_MIN;  // INT_MIN matches no entry
    }
    for (int i = tid; i < hn; i += kFusedThreads) s_hist[i] = 0;
    __syncthreads();

    // 2-3. earlier entries per own expert, and the histogram of experts [h0, h0 + hn)
    int own[KC], cnt[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      own[j] = j < a.k ? s_own[j] : INT_MIN;
      cnt[j] = 0;
    }
    auto visit = [&](int i, int e) {
      if (i < before) {
#pragma unroll
        for (int j = 0; j < KC; ++j) cnt[j] += e == own[j];
      }
      const unsigned hb = static_cast<unsigned>(e - h0);  // masked and invalid ids fall outside
      if (hb < static_cast<unsigned>(hn)) atomicAdd(&s_hist[hb], 1);
    };
    if (a.idx_vec) {
#pragma unroll
      for (int c = 0; c < kFusedScanRegs; ++c) {
        const int q = tid + c * kFusedThreads;
        if (4 * q < m) {
          visit(4 * q, r4[c].x);
          visit(4 * q + 1, r4[c].y);
          visit(4 * q + 2, r4[c].z);
          visit(4 * q + 3, r4[c].w);
        }
      }
      for (int q = tid + kFusedScanRegs * kFusedThreads; 4 * q < m; q += kFusedThreads) {
        const int4 e4 = __ldcg(reinterpret_cast<const int4 *>(ridx) + q);
        visit(4 * q, e4.x);
        visit(4 * q + 1, e4.y);
        visit(4 * q + 2, e4.z);
        visit(4 * q + 3, e4.w);
      }
    } else {
      for (int i = tid; i < m; i += kFusedThreads) visit(i, __ldcg(ridx + i));
    }
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      const int c = __reduce_add_sync(0xffffffffu, cnt[j]);
      if (lane == 0) s_part[warp][j] = c;
    }
    __syncthreads();

    // 4. the row's slots
    int32_t my_slot = -1;
    int my_e = 0;
    if (tid < a.k) {
      const int e = s_own[tid];
      if (e != INT_MIN) {
        int pos = 0;
#pragma unroll
        for (int w = 0; w < kFusedWarps; ++w) pos += s_part[w][tid];
        if (pos < a.max_m)
          my_slot = static_cast<int32_t>((static_cast<int64_t>(e) * a.R + src) * a.max_m + pos);
        else
          latch_error(a.err, MOE_EOVERFLOW);
        for (int j = 0; j < tid; ++j)
          if (s_own[j] == e) latch_error(a.err, MOE_EINVAL);  // expert repeated within the token
      } else if (__ldcg(own_p + tid) != kMaskedExpert) {
        latch_error(a.err, MOE_EINVAL);  // a masked choice is skipped silently
      }
      my_e = e;
      s_slot[tid] = my_slot;
      if (my_slot >= 0) {
        int g;
        const int64_t l = slot_local(a.parts, my_slot, &g);
        s_dst[tid] = a.parts.recv_x[g] + l * a.row_bytes;
        s_dsc[tid] = a.nsc > 0 ? a.parts.recv_scales[g] + l * a.nsc : nullptr;
      }
    }
    __syncthreads();

    // 5. the k copies
    const uint64_t pol = l2_evict_last_policy();
    if constexpr (!QUANT) {
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        if (j >= a.k) break;
        if (s_slot[j] < 0) continue;
        uint8_t *dst = s_dst[j];
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
          const int q = tid + u * kFusedThreads;
          if (q < a.vin) st_row<W>(dst + static_cast<int64_t>(q) * W, v[u], pol);
        }
        if (a.nsc > 0) {
          float *ds = s_dsc[j];
          if (a.sc_vec) {
            if (tid < a.nsc / 4) reinterpret_cast<float4 *>(ds)[tid] = sc;
          } else if (tid < a.nsc) {
            ds[tid] = sc.x;
          }
        }
      }
    } else {
      // Quantise on dispatch. Vector q holds bf16 elements (W/2)q .. (W/2)q +
      // W/2 - 1, so a 128-element block is G = 256 / W consecutive lanes (vin is
      // a multiple of G). scale = amax / 448 (1 for an all-zero block), code =
      // e4m3(x / scale): the code of the IEEE fp32 quotient under the hardware's
      // nearest-even saturating conversion, found without a division unless the
      // quotient sits near an e4m3 rounding boundary (e4m3x2_of_quotients); W/2
      // codes per thread.
      constexpr int NE = W / 2;         // bf16 elements per vector
      constexpr int G = 256 / W;        // lanes per 128-element block
#pragma unroll
      for (int u = 0; u < VPT; ++u) {
        const int q = tid + u * kFusedThreads;
        float f[NE];
#pragma unroll
        for (int p = 0; p < NE / 2; ++p) {
          f[2 * p] = __uint_as_float(v[u].w[p] << 16);
          f[2 * p + 1] = __uint_as_float(v[u].w[p] & 0xffff0000u);
        }
        float amax = 0.0f;
#pragma unroll
        for (int p = 0; p < NE; ++p) amax = fmaxf(amax, fabsf(f[p]));
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const BlockScale bs = block_scale(amax);
        const float s = bs.s;
        uint32_t c[NE / 4];
#pragma unroll
        for (int p = 0; p < NE / 4; ++p)
          c[p] = static_cast<uint32_t>(e4m3x2_of_quotients(f[4 * p], f[4 * p + 1], bs)) |
                 (static_cast<uint32_t>(e4m3x2_of_quotients(f[4 * p + 2], f[4 * p + 3], bs)) << 16);
        // 16-byte stores: 32-byte vectors give 16 codes each; 16-byte vectors
        // give 8, so even lanes take their odd neighbour's 8 as well
        RowVec<16> out16;
        bool store16;
        if constexpr (W == 32) {
          out16 = RowVec<16>{{c[0], c[1], c[2], c[3]}};
          store16 = true;
        } else {
          const uint32_t px = __shfl_xor_sync(0xffffffffu, c[0], 1);
          const uint32_t py = __shfl_xor_sync(0xffffffffu, c[1], 1);
          out16 = RowVec<16>{{c[0], c[1], px, py}};
          store16 = (q & 1) == 0;
        }
        if (q >= a.vin) continue;  // whole G-lane groups are out together
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          if (j >= a.k) break;
          if (s_slot[j] < 0) continue;
          uint8_t *dst = s_dst[j];
          if (store16) st_row<16>(dst + static_cast<int64_t>(q) * NE, out16, pol);
          if (q % G == 0) s_dsc[j][q / G] = s;
        }
      }
    }

    // 6. the step's records, after the copies (nothing above waits for them):
    //    tok_slot, the slot headers, and the counts and count + 1 flags of
    //    this row's share of the experts
    if (tid < a.k) {
      a.tok_slot[row * a.k + tid] = my_slot;
      if (my_slot >= 0) {
        int g;
        const int64_t l = slot_local(a.parts, my_slot, &g);
        a.parts.recv_meta[g][l] = make_int4(src, t, my_e, tid);
      }
    }
    for (int i = tid; i < hn; i += kFusedThreads) {
      const int c = s_hist[i];
      const int64_t r = static_cast<int64_t>(h0 + i) * a.R + src;
      a.counts[r] = c;
      *flag_ptr(a.parts, r) = static_cast<uint64_t>(c) + 1;
    }
    if (row + gridDim.x < a.nrows) __syncthreads();  // the next row reuses the shared arrays
  }
}

// Vectors per thread of the fused kernel (a power of two covering vin, at most
// max_vpt), or 0 when a row is too long.
static int fused_vpt(int64_t vin, int max_vpt) {
  const int64_t need = (vin + kFusedThreads - 1) / kFusedThreads;
  for (int p = 1; p <= max_vpt; p *= 2)
    if (need <= p) return p;
  return 0;
}

static int fused_hist(const Sizes &s) {
  const int rows = s.T < kFusedHistRows ? s.T : kFusedHistRows;
  return rows > 0 ? (s.E + rows - 1) / rows : s.E;
}

// Whether the batch runs as the one fused kernel (rows of at most 16 KiB).
static bool fused_fits(const Sizes &s) {
  if (s.ntok == 0 || s.T > kFusedMaxTokens || s.in_row_bytes % 16 != 0) return false;
  if (fused_vpt(s.in_row_bytes / 16, kFusedMaxVec16) == 0) return false;
  return fused_hist(s) <= kFusedMaxHist;
}

int layout_dispatch_kernel_count(const Sizes &s) { return (s.ntok == 0 || fused_fits(s)) ? 1 : 2; }

template <int W, int VPT, int KC, bool QUANT>
static moe_status launch_fused(const FusedArgs &a, int sms, cudaStream_t stream) {
  auto kern = layout_dispatch_kernel<W, VPT, KC, QUANT>;
  const size_t smem = static_cast<size_t>(a.G) * sizeof(int32_t);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return MOE_ECUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFusedThreads, smem) != cudaSuccess)
    return MOE_ECUDA;
  if (per_sm < 1) return MOE_EINVAL;
  // one row per CTA while every CTA is resident at once; beyond that, CTAs loop
  const int64_t capacity = static_cast<int64_t>(sms) * per_sm;
  const int64_t grid = a.nrows < capacity ? a.nrows : capacity;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

template <int KC, bool QUANT>
static moe_status launch_fused_w(const FusedArgs &a, int width, int sms, cudaStream_t stream) {
  if (width == 32) {
    switch (fused_vpt(a.vin, kFusedMaxVec32)) {
      case 1: return launch_fused<32, 1, KC, QUANT>(a, sms, stream);
      case 2: return launch_fused<32, 2, KC, QUANT>(a, sms, stream);
      case 4: return launch_fused<32, 4, KC, QUANT>(a, sms, stream);
      default: return MOE_EINVAL;
    }
  }
  if constexpr (!QUANT) {
    switch (fused_vpt(a.vin, kFusedMaxVec16)) {
      case 1: return launch_fused<16, 1, KC, false>(a, sms, stream);
      case 2: return launch_fused<16, 2, KC, false>(a, sms, stream);
      case 4: return launch_fused<16, 4, KC, false>(a, sms, stream);
      default: break;
    }
  }
  return launch_fused<16, 8, kMaxTopk, QUANT>(a, sms, stream);  // rows whose pointers allow only 16 bytes
}

moe_status launch_layout_dispatch(const Sizes &s, const int32_t *topk_idx, const void *x, const float *x_scales,
                                  int32_t *counts, int32_t *tok_slot, const SlotParts &parts, int32_t *err,
                                  int num_sms, cudaStream_t stream) {
  if (!fused_fits(s)) {
    moe_status st = launch_layout(s, topk_idx, counts, parts, tok_slot, err, stream);
    if (st != MOE_OK || s.ntok == 0) return st;
    return launch_dispatch(s, x, x_scales, tok_slot, parts, err, num_sms, stream);
  }
  // Vector width, measured on GB300: plain copies of rows up to 8 KiB are
  // fastest with 16-byte vectors (ds_decode step 36.6 vs 37.6 us with 32-byte
  // ones), longer rows and quantised rows with 32-byte vectors (skewed 162.3
  // vs 163.4 us; ds_decode with bf16 rows 46.1 vs 56.6 us), where the rows and
  // pointers allow them.
  bool rows32 = s.row_bytes % 32 == 0;
  bool scales16 = true;
  for (int g = 0; g < parts.G; ++g) {
    rows32 = rows32 && aligned32(parts.recv_x[g]);
    scales16 = scales16 && aligned16(parts.recv_scales[g]);
  }
  const bool can32 = s.in_row_bytes % 32 == 0 && aligned32(x) && (s.quant || rows32);
  const bool wide = can32 && (s.quant || s.in_row_bytes > kFusedNarrowMaxRow);
  FusedArgs a{};
  a.topk_idx = topk_idx;
  a.counts = counts;
  a.tok_slot = tok_slot;
  a.x = static_cast<const uint8_t *>(x);
  a.x_scales = x_scales;
  a.parts = parts;
  a.err = err;
  a.R = s.R;
  a.T = s.T;
  a.E = s.E;
  a.k = s.k;
  a.max_m = s.max_m;
  a.nsc = s.nsc;
  a.G = fused_hist(s);
  a.early = early_trigger(s.ntok);
  a.vin = static_cast<int>(s.in_row_bytes / (wide ? 32 : 16));
  a.idx_vec = (static_cast<int64_t>(s.T) * s.k) % 4 == 0 && aligned16(topk_idx) ? 1 : 0;
  a.sc_vec = s.nsc % 4 == 0 && aligned16(x_scales) && scales16 ? 1 : 0;
  a.row_bytes = static_cast<uint32_t>(s.row_bytes);
  a.in_row_bytes = static_cast<uint32_t>(s.in_row_bytes);
  a.nrows = s.ntok;
  const int sms = num_sms > 0 && num_sms < sm_count() ? num_sms : sm_count();
  const int width = wide ? 32 : 16;
  if (s.k <= 8)
    return s.quant ? launch_fused_w<8, true>(a, width, sms, stream) : launch_fused_w<8, false>(a, width, sms, stream);
  return s.quant ? launch_fused_w<kMaxTopk, true>(a, width, sms, stream)
                 : launch_fused_w<kMaxTopk, false>(a, width, sms, stream);
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_layout_dispatch(const moe_desc *desc, const int32_t *topk_idx, const void *x,
                                          const float *x_scales, int32_t *counts, uint64_t *flags,
                                          int32_t *tok_slot, void *recv_x, float *recv_scales,
                                          int32_t *recv_meta, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (counts == nullptr || flags == nullptr || err == nullptr || recv_x == nullptr || recv_meta == nullptr)
    return MOE_EINVAL;
  if (s.ntok > 0 && (topk_idx == nullptr || tok_slot == nullptr || x == nullptr)) return MOE_EINVAL;
  if (s.dtype == MOE_FP8_E4M3) {
    if (recv_scales == nullptr || (s.ntok > 0 && x_scales == nullptr)) return MOE_EINVAL;
    if (!aligned4(x_scales) || !aligned4(recv_scales)) return MOE_EINVAL;
  } else if (s.dtype == MOE_BF16_TO_FP8) {
    if (recv_scales == nullptr || x_scales != nullptr || !aligned4(recv_scales)) return MOE_EINVAL;
  }
  if (!aligned16(x) || !aligned16(recv_x) || !aligned16(recv_meta) || !aligned4(tok_slot) || !aligned4(err) ||
      !aligned4(topk_idx) || !aligned4(counts) || (reinterpret_cast<uintptr_t>(flags) & 7u) != 0)
    return MOE_EINVAL;
  return launch_layout_dispatch(s, topk_idx, x, x_scales, counts, tok_slot,
                                single_part(s, recv_x, recv_scales, recv_meta, flags, nullptr), err, desc->num_sms,
                                static_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_layout_dispatch_parts(const moe_desc *desc, const int32_t *topk_idx, const void *x,
                                                const float *x_scales, int32_t *counts, int32_t *tok_slot,
                                                const moe_parts *parts, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  SlotParts p;
  st = parts_from(s, parts, true, false, &p);
  if (st != MOE_OK) return st;
  if (counts == nullptr || err == nullptr) return MOE_EINVAL;
  if (s.ntok > 0 && (topk_idx == nullptr || tok_slot == nullptr || x == nullptr)) return MOE_EINVAL;
  if (s.dtype == MOE_FP8_E4M3 && (s.ntok > 0 && x_scales == nullptr)) return MOE_EINVAL;
  if (s.dtype != MOE_FP8_E4M3 && x_scales != nullptr) return MOE_EINVAL;
  if (!aligned16(x) || !aligned4(x_scales) || !aligned4(tok_slot) || !aligned4(err) || !aligned4(topk_idx) ||
      !aligned4(counts))
    return MOE_EINVAL;
  return launch_layout_dispatch(s, topk_idx, x, x_scales, counts, tok_slot, p, err, desc->num_sms,
                                static_cast<cudaStream_t>(stream));
}

extern "C" int32_t moe_layout_dispatch_kernels(const moe_desc *desc) {
  Sizes s;
  if (check_desc(desc, &s) != MOE_OK) return MOE_EINVAL;
  return layout_dispatch_kernel_count(s);
}

// Layout and dispatch in one kernel, for batches whose per-rank routing fits
// one CTA's shared memory (decode-sized batches).
//
// Same results as moe_layout followed by moe_dispatch (Perplexity,
// "Efficient and portable mixture-of-experts communication", section
// "Dispatch": one warp counts the tokens per destination expert while the
// other warps pack the tokens; "NVSHMEM and DeepEP: GPU-initiated
// communication", low-latency section: fixed slots, no exchange). Here every
// CTA is such a sender for a few rows of one source rank:
//   - thread 0 starts the bulk TMA loads of its rows (x is an input, so this
//     happens before waiting on the previous kernel);
//   - all threads build the per-expert token bitmaps of the whole source rank
//     (T bits per expert, T <= 1024) from topk_idx, which gives every count and
//     every token-order slot position locally, with no grid-wide step and no
//     wait on another CTA;
//   - the CTA writes its rows' tok_slot entries, headers and scales, and thread
//     0 writes each staged row into its k slots with bulk TMA stores;
//   - the first CTA of each source rank writes counts and count + 1 flags.
// A sender computes its own counts, so it needs no flag wait; the flags are
// still written for the consumers of the step.
#include "moe_common.cuh"

namespace moe {

constexpr int kFusedThreads = 128;
constexpr int kFusedMaxTokens = 1024;
constexpr uint32_t kFusedMaxRowBytes = 16384;
constexpr size_t kFusedMaxSmem = 96 * 1024;

struct FusedArgs {
  const int32_t *topk_idx;
  int32_t *counts;
  uint64_t *flags;
  int32_t *tok_slot;
  const uint8_t *x;
  const float *x_scales;
  uint8_t *recv_x;
  float *recv_scales;
  int4 *recv_meta;
  int32_t *err;
  int R, T, E, k, max_m, nsc, words, ctas_per_rank, stages, early, quant;
  uint32_t row_bytes;     // a dispatched row (the slot stride)
  uint32_t in_row_bytes;  // a caller's input row (the stage size)
  uint32_t qoff;          // quant mode: offset of the e4m3 row buffer in shared memory
  int64_t nslots;
};

__global__ void __launch_bounds__(kFusedThreads) layout_dispatch_kernel(FusedArgs a) {
  extern __shared__ __align__(128) uint8_t fsm[];
  __shared__ uint64_t full[kMaxStages];
  __shared__ int32_t dst[kMaxTopk];
  __shared__ int aborted;

  const int tid = threadIdx.x;
  const int src = blockIdx.x / a.ctas_per_rank;
  const int c = blockIdx.x % a.ctas_per_rank;
  const int S = a.stages;
  // rows t = c, c + C, c + 2C, ... of source rank src
  const int n_mine = c < a.T ? (a.T - 1 - c) / a.ctas_per_rank + 1 : 0;
  uint32_t *bits = reinterpret_cast<uint32_t *>(fsm + static_cast<size_t>(S) * a.in_row_bytes);
  const uint8_t *xs = a.x + static_cast<int64_t>(src) * a.T * a.in_row_bytes;
  uint8_t *qbuf = fsm + a.qoff;                                   // quant mode: e4m3 row
  float *qsc = reinterpret_cast<float *>(fsm + a.qoff + a.row_bytes);  // quant mode: its scales

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    aborted = 0;
    for (int i = 0; i < n_mine && i < S; ++i) {
      const int t = c + i * a.ctas_per_rank;
      mbar_arrive_expect_tx(&full[i], a.in_row_bytes);
      bulk_load(fsm + static_cast<size_t>(i) * a.in_row_bytes, xs + static_cast<int64_t>(t) * a.in_row_bytes,
                a.in_row_bytes, &full[i]);
    }
  }
  grid_dependency_wait();
  if (a.early) grid_dependents_launch();

  // per-expert token bitmaps of the whole source rank
  for (int i = tid; i < a.E * a.words; i += kFusedThreads) bits[i] = 0;
  __syncthreads();
  const int32_t *idx = a.topk_idx + static_cast<int64_t>(src) * a.T * a.k;
  for (int i = tid; i < a.T * a.k; i += kFusedThreads) {
    const int e = __ldg(idx + i);
    if (e < 0 || e >= a.E) {
      if (e != kMaskedExpert) latch_error(a.err, MOE_EINVAL);  // a masked choice is skipped silently
      continue;
    }
    const int t = i / a.k;
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&bits[e * a.words + (t >> 5)], bit) & bit) latch_error(a.err, MOE_EINVAL);
  }
  __syncthreads();

  if (c == 0) {
    for (int e = tid; e < a.E; e += kFusedThreads) {
      int cnt = 0;
      for (int w = 0; w < a.words; ++w) cnt += __popc(bits[e * a.words + w]);
      const int64_t r = static_cast<int64_t>(e) * a.R + src;
      a.counts[r] = cnt;
      a.flags[r] = static_cast<uint64_t>(cnt) + 1;
    }
  }

  int i = 0;
  for (; i < n_mine; ++i) {
    const int s = i % S;
    const uint32_t parity = static_cast<uint32_t>((i / S) & 1);
    const int t = c + i * a.ctas_per_rank;
    const int64_t row = static_cast<int64_t>(src) * a.T + t;
    if (tid < a.k) {
      const int e = __ldg(idx + t * a.k + tid);
      int32_t slot = -1;
      if (e >= 0 && e < a.E) {
        const uint32_t *b = bits + e * a.words;
        int pos = 0;
        for (int w = 0; w < (t >> 5); ++w) pos += __popc(b[w]);
        pos += __popc(b[t >> 5] & ((1u << (t & 31)) - 1u));
        if (pos < a.max_m)
          slot = static_cast<int32_t>((static_cast<int64_t>(e) * a.R + src) * a.max_m + pos);
        else
          latch_error(a.err, MOE_EOVERFLOW);
      }
      a.tok_slot[row * a.k + tid] = slot;
      dst[tid] = slot;
      if (slot >= 0) a.recv_meta[slot] = make_int4(src, t, e, tid);
    }
    __syncthreads();
    if (a.quant) {
      uint8_t *stage = fsm + static_cast<size_t>(s) * a.in_row_bytes;
      if (!mbar_wait_bounded(&full[s], parity)) {  // every thread reads the staged bf16 row
        latch_error(a.err, MOE_ETIMEOUT);
        aborted = 1;
      }
      if (tid == 0 && i > 0) bulk_wait_read<0>();  // the previous row's stores may still read qbuf
      __syncthreads();
      if (aborted) break;
      quantize_blocks(reinterpret_cast<const uint16_t *>(stage), qbuf, qsc, a.nsc, tid >> 5, kFusedThreads / 32,
                      tid & 31);
      fence_proxy_async_smem();  // the shared writes above, before the bulk stores and the refill
      __syncthreads();
      for (int q = tid; q < a.k * a.nsc; q += kFusedThreads) {
        const int j = q / a.nsc, cc = q - j * a.nsc;
        const int32_t slot = dst[j];
        if (slot >= 0) a.recv_scales[static_cast<int64_t>(slot) * a.nsc + cc] = qsc[cc];
      }
      if (tid == 0) {
        for (int j = 0; j < a.k; ++j)
          if (dst[j] >= 0) bulk_store(a.recv_x + static_cast<int64_t>(dst[j]) * a.row_bytes, qbuf, a.row_bytes);
        bulk_commit();
        if (i + S < n_mine) {  // the bf16 stage has been consumed: refill it with row i + S
          const int tn = c + (i + S) * a.ctas_per_rank;
          mbar_arrive_expect_tx(&full[s], a.in_row_bytes);
          bulk_load(stage, xs + static_cast<int64_t>(tn) * a.in_row_bytes, a.in_row_bytes, &full[s]);
        }
      }
      __syncthreads();
      continue;
    }
    if (a.nsc > 0) {
      const float *sc = a.x_scales + row * a.nsc;
      for (int q = tid; q < a.k * a.nsc; q += kFusedThreads) {
        const int j = q / a.nsc, cc = q - j * a.nsc;
        const int32_t slot = dst[j];
        if (slot >= 0) a.recv_scales[static_cast<int64_t>(slot) * a.nsc + cc] = __ldg(sc + cc);
      }
    }
    if (tid == 0) {
      uint8_t *stage = fsm + static_cast<size_t>(s) * a.in_row_bytes;
      if (!mbar_wait_bounded(&full[s], parity)) {
        latch_error(a.err, MOE_ETIMEOUT);
        aborted = 1;
      } else {
        for (int j = 0; j < a.k; ++j)
          if (dst[j] >= 0) bulk_store(a.recv_x + static_cast<int64_t>(dst[j]) * a.row_bytes, stage, a.row_bytes);
        bulk_commit();
        const int next = i - 1 + S;
        if (i >= 1 && next < n_mine) {
          bulk_wait_read<1>();
          const int ps = (i - 1) % S;
          const int tn = c + next * a.ctas_per_rank;
          mbar_arrive_expect_tx(&full[ps], a.in_row_bytes);
          bulk_load(fsm + static_cast<size_t>(ps) * a.in_row_bytes, xs + static_cast<int64_t>(tn) * a.in_row_bytes,
                    a.in_row_bytes, &full[ps]);
        }
      }
    }
    __syncthreads();
    if (aborted) break;
  }
  if (tid == 0) {
    if (aborted) {
      // drain the loads still in flight (bounded) before the CTA releases its shared memory
      const int issued = a.quant ? min(n_mine, i + S) : static_cast<int>(inflight_end(i, S, n_mine));
      for (int u = i; u < issued; ++u) mbar_wait_bounded(&full[u % S], static_cast<uint32_t>((u / S) & 1));
    }
    bulk_wait_all();
  }
}

// Offset of the e4m3 row buffer (quant mode): after the row stages and the bitmaps.
static size_t fused_qoff(const Sizes &s, int stages) {
  const int words = (s.T + 31) / 32;
  const size_t end = static_cast<size_t>(stages) * s.in_row_bytes + static_cast<size_t>(s.E) * (words > 0 ? words : 1) * 4;
  return (end + 127) / 128 * 128;
}

// Whether one CTA can hold a source rank's bitmaps next to its row stages.
static bool fused_fits(const Sizes &s, int stages, size_t *smem) {
  if (s.T > kFusedMaxTokens || s.in_row_bytes > kFusedMaxRowBytes || s.in_row_bytes % 16 != 0) return false;
  const int words = (s.T + 31) / 32;
  *smem = static_cast<size_t>(stages) * s.in_row_bytes + static_cast<size_t>(s.E) * (words > 0 ? words : 1) * 4;
  if (s.quant) *smem = fused_qoff(s, stages) + static_cast<size_t>(s.row_bytes) + static_cast<size_t>(s.nsc) * 4;
  return *smem <= kFusedMaxSmem;
}

int layout_dispatch_kernel_count(const Sizes &s) {
  size_t smem = 0;
  return (s.ntok == 0 || !fused_fits(s, 2, &smem)) ? (s.ntok == 0 ? 1 : 2) : 1;
}

moe_status launch_layout_dispatch(const Sizes &s, const int32_t *topk_idx, const void *x, const float *x_scales,
                                  int32_t *counts, uint64_t *flags, int32_t *tok_slot, void *recv_x,
                                  float *recv_scales, int32_t *recv_meta, int32_t *err, int num_sms,
                                  cudaStream_t stream) {
  size_t smem = 0;
  if (s.ntok == 0 || !fused_fits(s, 2, &smem)) {
    moe_status st = launch_layout(s, topk_idx, counts, flags, tok_slot, err, stream);
    if (st != MOE_OK) return st;
    return launch_dispatch(s, x, x_scales, tok_slot, flags, recv_x, recv_scales, recv_meta, err, num_sms, stream);
  }
  FusedArgs a{};
  a.topk_idx = topk_idx;
  a.counts = counts;
  a.flags = flags;
  a.tok_slot = tok_slot;
  a.x = static_cast<const uint8_t *>(x);
  a.x_scales = x_scales;
  a.recv_x = static_cast<uint8_t *>(recv_x);
  a.recv_scales = recv_scales;
  a.recv_meta = reinterpret_cast<int4 *>(recv_meta);
  a.err = err;
  a.R = s.R;
  a.T = s.T;
  a.E = s.E;
  a.k = s.k;
  a.max_m = s.max_m;
  a.nsc = s.nsc;
  a.words = (s.T + 31) / 32;
  a.early = early_trigger(s.ntok);
  a.quant = s.quant ? 1 : 0;
  a.row_bytes = static_cast<uint32_t>(s.row_bytes);
  a.in_row_bytes = static_cast<uint32_t>(s.in_row_bytes);
  a.nslots = s.nslots;

  const int sms = num_sms > 0 && num_sms < sm_count() ? num_sms : sm_count();
  // first try one row per CTA (one stage); with fewer CTAs than rows use two stages
  for (int stages = 1; stages <= 2; ++stages) {
    if (!fused_fits(s, stages, &smem)) return MOE_EINVAL;
    a.qoff = static_cast<uint32_t>(fused_qoff(s, stages));
    if (smem > 48 * 1024 && cudaFuncSetAttribute(layout_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem)) != cudaSuccess)
      return MOE_ECUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layout_dispatch_kernel, kFusedThreads, smem) !=
        cudaSuccess)
      return MOE_ECUDA;
    if (per_sm < 1) return MOE_EINVAL;
    const int64_t capacity = static_cast<int64_t>(sms) * per_sm;
    int64_t per_rank = capacity / s.R;
    if (per_rank < 1) per_rank = 1;
    if (per_rank > s.T) per_rank = s.T;
    const int rows = static_cast<int>((s.T + per_rank - 1) / per_rank);
    if (rows > 1 && stages == 1) continue;
    a.ctas_per_rank = static_cast<int>(per_rank);
    a.stages = stages;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(per_rank * s.R), 1, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    use_pdl(cfg, attr);
    if (cudaLaunchKernelEx(&cfg, layout_dispatch_kernel, a) != cudaSuccess) return MOE_ECUDA;
    return launch_status();
  }
  return MOE_EINVAL;
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
  return launch_layout_dispatch(s, topk_idx, x, x_scales, counts, flags, tok_slot, recv_x, recv_scales, recv_meta,
                                err, desc->num_sms, static_cast<cudaStream_t>(stream));
}

extern "C" int32_t moe_layout_dispatch_kernels(const moe_desc *desc) {
  Sizes s;
  if (check_desc(desc, &s) != MOE_OK) return MOE_EINVAL;
  return layout_dispatch_kernel_count(s);
}

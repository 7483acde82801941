// Combine (K3): for every token, the router-weighted sum of its k expert
// outputs, gathered through the slot ids that layout assigned.
//
// "How GPUs Talk to Each Other During LLM Inference", section 7: each expert
// output is weighted by the router's score for that expert and the k outputs
// of a token are added up at the token's home. Perplexity, "Efficient and
// portable mixture-of-experts communication", section "Combine": the receiver
// reads each payload from the private buffer the routing table points at,
// applies that expert's weight and writes the sum into a caller tensor; the
// combine is also the step's only barrier. "NVSHMEM and DeepEP", high-throughput
// section: combine returns BF16.
//
// Design: the work is (token, 16-byte column vector) tasks, 8 bf16 each. A
// block of 128 threads covers 128*VPT consecutive vectors of one token; each
// thread loads the token's k slot ids and weights (warp-broadcast loads), issues
// all k x VPT streaming 16-byte loads of its vectors first, then forms w_0*y_0
// and adds w_j*y_j in fp32 with FMA in choice order j = 1..k-1 (the sum starts
// from its first term, so signed zeros survive) and stores bf16 (round to
// nearest even) with a streaming store. The grid is all tasks, so waves of
// blocks overlap and keep enough bytes in flight to cover HBM latency. Pure
// HBM gather: no tensor cores, no shared memory. Block 0 also clears the
// count+1 flags: dispatch, their only reader, finished before this kernel in
// stream order, so the next layout signals afresh.
#include <cuda_bf16.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kCombineThreads = 128;

struct CombineArgs {
  SlotParts parts;  // the expert outputs y (rows of H) and the count + 1 flags, per part
  const float *weights;
  const int32_t *tok_slot;
  uint16_t *out;
  int32_t *err;
  int H, k, chunks, early;
  int64_t nslots;  // rows of y: the slots (fixed-slot layout) or the packed rows
};

// Row `slot` of y, in its part (PARTS: more than one part; one part is the
// single buffer, with the address arithmetic of a plain array).
template <bool PARTS>
__device__ __forceinline__ const uint16_t *y_row(const CombineArgs &a, int32_t slot) {
  if constexpr (!PARTS) return a.parts.y[0] + static_cast<int64_t>(slot) * a.H;
  int g;
  const int64_t l = slot_local(a.parts, slot, &g);
  return a.parts.y[g] + l * a.H;
}

// Block b < G clears part b's count + 1 flags.
__device__ __forceinline__ void clear_flags(const CombineArgs &a, int64_t b) {
  if (b < a.parts.G)
    for (int i = threadIdx.x; i < a.parts.regions_per_part; i += blockDim.x) a.parts.flags[b][i] = 0;
}

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4 &v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = fmaf(w, __uint_as_float(u[q] << 16), acc[2 * q]);
    acc[2 * q + 1] = fmaf(w, __uint_as_float(u[q] & 0xffff0000u), acc[2 * q + 1]);
  }
}

__device__ __forceinline__ void mul_bf16x8(float (&acc)[8], float w, const uint4 &v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = __fmul_rn(w, __uint_as_float(u[q] << 16));
    acc[2 * q + 1] = __fmul_rn(w, __uint_as_float(u[q] & 0xffff0000u));
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
  uint32_t u[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
    u[q] = *reinterpret_cast<uint32_t *>(&p);
  }
  return make_uint4(u[0], u[1], u[2], u[3]);
}

// Large batches (at least kCombineTmaMinTokens tokens, k >= 4): thread 0
// stages the k pieces (128 vectors of 16 bytes each) of a (token, column
// chunk) task in shared memory with bulk TMA loads on one mbarrier, and every
// thread combines its vector from shared memory. Measured on GB300: faster than
// the register gather for the 32768-token DeepSeek-shape prefill (592 vs
// 668 us per combine inside the step), slower for decode-sized batches.
constexpr int64_t kCombineTmaMinTokens = 16384;

template <int K, bool PARTS>
__global__ void __launch_bounds__(kCombineThreads) combine_tma_kernel(CombineArgs a) {
  __shared__ __align__(128) uint4 stage[K][kCombineThreads];
  __shared__ uint64_t bar;
  __shared__ int32_t s_slot[K];
  __shared__ float s_w[K];
  const int64_t b = blockIdx.x;
  const int64_t tok = b / a.chunks;
  const int V = a.H / 8;
  const int v0 = static_cast<int>(b % a.chunks) * kCombineThreads;
  const int nv = min(kCombineThreads, V - v0);
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  grid_dependency_wait();
  if (a.early) grid_dependents_launch();
  clear_flags(a, b);
  if (tid < K) {
    int32_t slot = __ldg(a.tok_slot + tok * K + tid);
    float w = __ldg(a.weights + tok * K + tid);
    if (slot >= a.nslots) {
      latch_error(a.err, MOE_EINVAL);
      slot = -1;
    }
    if (slot < 0) w = 0.0f;  // an entry layout rejected contributes nothing
    s_slot[tid] = slot;
    s_w[tid] = w;
  }
  __syncthreads();
  if (tid == 0) {
    int nvalid = 0;
    for (int j = 0; j < K; ++j) nvalid += s_slot[j] >= 0;
    const uint32_t bytes = static_cast<uint32_t>(nv) * 16;
    mbar_arrive_expect_tx(&bar, nvalid * bytes);
    for (int j = 0; j < K; ++j)
      if (s_slot[j] >= 0)
        bulk_load(&stage[j][0], y_row<PARTS>(a, s_slot[j]) + static_cast<int64_t>(v0) * 8, bytes,
                  &bar);
  }
  if (!mbar_wait_bounded(&bar, 0)) {
    latch_error(a.err, MOE_ETIMEOUT);
    mbar_wait_bounded(&bar, 0);  // drain (bounded) before the shared memory is released
    return;
  }
  if (tid < nv) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    // the sum of the k terms starts from the first term (an all -0 token stays -0)
    float acc[8];
    mul_bf16x8(acc, s_w[0], s_slot[0] >= 0 ? stage[0][tid] : zero);
#pragma unroll
    for (int j = 1; j < K; ++j) fma_bf16x8(acc, s_w[j], s_slot[j] >= 0 ? stage[j][tid] : zero);
    __stcs(reinterpret_cast<uint4 *>(a.out + tok * a.H) + v0 + tid, pack_bf16x8(acc));
  }
}

// K > 0: compile-time number of choices; K == 0: runtime k (<= kMaxTopk).
// Block b handles token b / chunks, column vectors [c*128*VPT, (c+1)*128*VPT)
// with c = b % chunks; each thread owns VPT vectors and issues all their k
// loads before it computes.
template <int K, int VPT, bool PARTS>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs a) {
  constexpr int KC = K > 0 ? K : kMaxTopk;
  const int k = K > 0 ? K : a.k;
  const int64_t b = blockIdx.x;
  const int64_t tok = b / a.chunks;
  const int v0 = static_cast<int>(b % a.chunks) * kCombineThreads * VPT + threadIdx.x;
  const int V = a.H / 8;

  grid_dependency_wait();
  if (a.early) grid_dependents_launch();
  clear_flags(a, b);

  // this token's slots and weights (the same for the whole warp: broadcast loads)
  int32_t slot[KC];
  float w[KC];
#pragma unroll
  for (int j = 0; j < KC; ++j) {
    if (j < k) {
      slot[j] = __ldg(a.tok_slot + tok * k + j);
      w[j] = __ldg(a.weights + tok * k + j);
      if (slot[j] >= a.nslots) {
        latch_error(a.err, MOE_EINVAL);
        slot[j] = -1;
      }
      if (slot[j] < 0) w[j] = 0.0f;  // an entry layout rejected contributes nothing
    }
  }

  uint4 y[VPT][KC];
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const int v = v0 + u * kCombineThreads;
#pragma unroll
    for (int j = 0; j < KC; ++j)
      if (j < k)
        y[u][j] = (v < V && slot[j] >= 0)
                      ? __ldcs(reinterpret_cast<const uint4 *>(y_row<PARTS>(a, slot[j])) + v)
                      : make_uint4(0, 0, 0, 0);
  }
  uint4 *dst = reinterpret_cast<uint4 *>(a.out + tok * a.H);
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const int v = v0 + u * kCombineThreads;
    if (v >= V) break;
    // the sum of the k terms starts from the first term (an all -0 token stays -0)
    float acc[8];
    mul_bf16x8(acc, w[0], y[u][0]);
#pragma unroll
    for (int j = 1; j < KC; ++j)
      if (j < k) fma_bf16x8(acc, w[j], y[u][j]);
    __stcs(dst + v, pack_bf16x8(acc));
  }
}

template <int K, int VPT>
moe_status launch_combine_k(CombineArgs a, int64_t ntok, cudaStream_t stream) {
  const int V = a.H / 8;
  const bool tma = K >= 4 && ntok >= kCombineTmaMinTokens;
  const int vpt = tma ? 1 : VPT;
  a.chunks = (V + kCombineThreads * vpt - 1) / (kCombineThreads * vpt);
  const int64_t blocks = ntok * a.chunks;
  if (blocks > 0x7fffffffll) return MOE_EINVAL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  const bool parts = a.parts.G > 1;
  if constexpr (K >= 4) {
    if (tma) {
      if (cudaLaunchKernelEx(&cfg, parts ? combine_tma_kernel<K, true> : combine_tma_kernel<K, false>, a) !=
          cudaSuccess)
        return MOE_ECUDA;
      return launch_status();
    }
  }
  if (cudaLaunchKernelEx(&cfg, parts ? combine_kernel<K, VPT, true> : combine_kernel<K, VPT, false>, a) !=
      cudaSuccess)
    return MOE_ECUDA;
  return launch_status();
}

moe_status launch_combine(const Sizes &s, const SlotParts &parts, int64_t y_rows, const float *weights,
                          const int32_t *tok_slot, uint16_t *out, int32_t *err, cudaStream_t stream) {
  CombineArgs a{parts, weights, tok_slot, out, err, s.H, s.k, 1, early_trigger(s.ntok), y_rows};
  if (s.ntok == 0) {
    // nothing to gather; still clear the flags for the next step
    for (int g = 0; g < parts.G; ++g)
      if (cudaMemsetAsync(parts.flags[g], 0, static_cast<size_t>(parts.regions_per_part) * sizeof(uint64_t),
                          stream) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
  }
  switch (s.k) {
    case 1: return launch_combine_k<1, 2>(a, s.ntok, stream);
    case 2: return launch_combine_k<2, 2>(a, s.ntok, stream);
    case 4: return launch_combine_k<4, 1>(a, s.ntok, stream);
    case 6: return launch_combine_k<6, 1>(a, s.ntok, stream);
    case 8: return launch_combine_k<8, 1>(a, s.ntok, stream);
    default: return launch_combine_k<0, 1>(a, s.ntok, stream);
  }
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_combine(const moe_desc *desc, const uint16_t *expert_out, const float *topk_weights,
                                  const int32_t *tok_slot, uint64_t *flags, uint16_t *out, int32_t *err,
                                  void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (flags == nullptr || err == nullptr) return MOE_EINVAL;
  if (s.ntok > 0 && (expert_out == nullptr || topk_weights == nullptr || tok_slot == nullptr || out == nullptr))
    return MOE_EINVAL;
  if (!aligned16(expert_out) || !aligned16(out) || !aligned4(topk_weights) || !aligned4(tok_slot) ||
      !aligned4(err) || (reinterpret_cast<uintptr_t>(flags) & 7u) != 0)
    return MOE_EINVAL;
  return launch_combine(s, single_part(s, nullptr, nullptr, nullptr, flags, expert_out), s.nslots, topk_weights,
                        tok_slot, out, err, static_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_combine_packed(const moe_desc *desc, const uint16_t *packed_y, const int32_t *tok_packed,
                                         const float *topk_weights, uint64_t *flags, uint16_t *out, int32_t *err,
                                         void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (flags == nullptr || err == nullptr) return MOE_EINVAL;
  if (s.ntok > 0 && (packed_y == nullptr || topk_weights == nullptr || tok_packed == nullptr || out == nullptr))
    return MOE_EINVAL;
  if (!aligned16(packed_y) || !aligned16(out) || !aligned4(topk_weights) || !aligned4(tok_packed) ||
      !aligned4(err) || (reinterpret_cast<uintptr_t>(flags) & 7u) != 0)
    return MOE_EINVAL;
  return launch_combine(s, single_part(s, nullptr, nullptr, nullptr, flags, packed_y), s.ntok * s.k, topk_weights,
                        tok_packed, out, err, static_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_combine_parts(const moe_desc *desc, const moe_parts *parts, const float *topk_weights,
                                        const int32_t *tok_slot, uint16_t *out, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  SlotParts p;
  st = parts_from(s, parts, false, s.ntok > 0, &p);
  if (st != MOE_OK) return st;
  if (err == nullptr) return MOE_EINVAL;
  if (s.ntok > 0 && (topk_weights == nullptr || tok_slot == nullptr || out == nullptr)) return MOE_EINVAL;
  if (!aligned16(out) || !aligned4(topk_weights) || !aligned4(tok_slot) || !aligned4(err)) return MOE_EINVAL;
  return launch_combine(s, p, s.nslots, topk_weights, tok_slot, out, err, static_cast<cudaStream_t>(stream));
}

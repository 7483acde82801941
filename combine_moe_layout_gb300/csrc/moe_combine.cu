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
// Design: one CTA of 128 threads per token; thread v handles 16-byte column
// vectors v, v+128, ... of the row (8 bf16). For each vector it issues all k
// streaming loads first (k x 16 B in flight per thread), then forms
// w_0 * y_0 and adds w_j * y_j in fp32 with FMA in choice order j = 1..k-1
// (the sum starts from its first term, so signed zeros survive), and stores the bf16
// (round to nearest even) result with a streaming store. Pure HBM gather:
// no tensor cores, no shared-memory staging. Block 0 also clears the count+1
// flags: dispatch, their only reader, finished before this kernel in stream
// order, so the next layout signals afresh.
#include <cuda_bf16.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kCombineThreads = 128;

struct CombineArgs {
  const uint16_t *y;
  const float *weights;
  const int32_t *tok_slot;
  uint64_t *flags;
  uint16_t *out;
  int32_t *err;
  int H, k, nflags;
  int64_t nslots;
};

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

// K > 0: compile-time number of choices; K == 0: runtime k (<= kMaxTopk).
template <int K>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs a) {
  constexpr int KC = K > 0 ? K : kMaxTopk;
  __shared__ int32_t s_slot[KC];
  __shared__ float s_w[KC];
  const int k = K > 0 ? K : a.k;
  const int64_t tok = blockIdx.x;
  const int tid = threadIdx.x;

  grid_dependency_wait();
  if (blockIdx.x == 0)
    for (int i = tid; i < a.nflags; i += blockDim.x) a.flags[i] = 0;

  if (tid < k) {
    int32_t slot = __ldg(a.tok_slot + tok * k + tid);
    float w = __ldg(a.weights + tok * k + tid);
    if (slot >= a.nslots) {
      latch_error(a.err, MOE_EINVAL);
      slot = -1;
    }
    if (slot < 0) w = 0.0f;  // an entry layout rejected contributes nothing
    s_slot[tid] = slot;
    s_w[tid] = w;
  }
  __syncthreads();

  const int V = a.H / 8;
  const uint4 *src[KC];
  float w[KC];
#pragma unroll
  for (int j = 0; j < KC; ++j) {
    if (j < k) {
      const int32_t slot = s_slot[j];
      src[j] = reinterpret_cast<const uint4 *>(a.y + static_cast<int64_t>(slot < 0 ? 0 : slot) * a.H);
      w[j] = s_w[j];
    }
  }
  uint4 *dst = reinterpret_cast<uint4 *>(a.out + tok * a.H);

  for (int v = tid; v < V; v += kCombineThreads) {
    uint4 y[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j)
      if (j < k) y[j] = s_slot[j] >= 0 ? __ldcs(src[j] + v) : make_uint4(0, 0, 0, 0);
    // the sum of the k terms starts from the first term (an all -0 token stays -0)
    float acc[8];
    mul_bf16x8(acc, w[0], y[0]);
#pragma unroll
    for (int j = 1; j < KC; ++j)
      if (j < k) fma_bf16x8(acc, w[j], y[j]);
    __stcs(dst + v, pack_bf16x8(acc));
  }
  grid_dependents_launch();
}

template <int K>
moe_status launch_combine_k(const CombineArgs &a, int64_t ntok, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ntok), 1, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, combine_kernel<K>, a) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

moe_status launch_combine(const Sizes &s, const uint16_t *y, const float *weights, const int32_t *tok_slot,
                          uint64_t *flags, uint16_t *out, int32_t *err, cudaStream_t stream) {
  CombineArgs a{y, weights, tok_slot, flags, out, err, s.H, s.k, s.E * s.R, s.nslots};
  if (s.ntok == 0) {
    // nothing to gather; still clear the flags for the next step
    if (cudaMemsetAsync(flags, 0, static_cast<size_t>(s.E) * s.R * sizeof(uint64_t), stream) != cudaSuccess)
      return MOE_ECUDA;
    return MOE_OK;
  }
  switch (s.k) {
    case 1: return launch_combine_k<1>(a, s.ntok, stream);
    case 2: return launch_combine_k<2>(a, s.ntok, stream);
    case 4: return launch_combine_k<4>(a, s.ntok, stream);
    case 6: return launch_combine_k<6>(a, s.ntok, stream);
    case 8: return launch_combine_k<8>(a, s.ntok, stream);
    default: return launch_combine_k<0>(a, s.ntok, stream);
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
  return launch_combine(s, expert_out, topk_weights, tok_slot, flags, out, err, static_cast<cudaStream_t>(stream));
}

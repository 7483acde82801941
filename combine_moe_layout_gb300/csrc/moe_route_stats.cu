// Cross-node traffic of a routing: per-node deduplication accounting.
//
// "NVSHMEM and DeepEP: GPU-initiated communication", high-throughput section:
// a token goes to the nodes of its k experts; the copies that leave its home
// node, counted per expert, per distinct destination GPU or per distinct
// destination node (DeepEP's per-node deduplication), measure the cross-node
// traffic of the three schemes. Node-limited routing lowers the last one.
//
// One CTA per source rank: each thread accumulates its tokens' three counts
// (k <= 16 choices, first-occurrence tests in registers), then a block
// reduction writes the rank's totals; no atomics, so no output needs zeroing.
#include "moe_common.cuh"

namespace moe {

constexpr int kStatsThreads = 256;

struct StatsArgs {
  const int32_t *topk_idx;
  int64_t *stats;
  int32_t *err;
  int T, E, k, L, ranks_per_node;
};

__global__ void __launch_bounds__(kStatsThreads) route_stats_kernel(StatsArgs a) {
  __shared__ int64_t red[3][kStatsThreads / 32];
  const int src = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int home = src / a.ranks_per_node;
  grid_dependency_wait();
  int64_t c[3] = {0, 0, 0};
  for (int t = tid; t < a.T; t += kStatsThreads) {
    const int32_t *row = a.topk_idx + (static_cast<int64_t>(src) * a.T + t) * a.k;
    int rank[kMaxTopk];
    for (int j = 0; j < a.k; ++j) {
      const int e = __ldg(row + j);
      if (e < 0 || e >= a.E) {
        if (e != kMaskedExpert) latch_error(a.err, MOE_EINVAL);  // a masked choice sends nothing
        rank[j] = -1;
        continue;
      }
      rank[j] = e / a.L;
      const int node = rank[j] / a.ranks_per_node;
      if (node == home) continue;
      bool seen_rank = false, seen_node = false;
      for (int jj = 0; jj < j; ++jj) {
        if (rank[jj] < 0) continue;
        seen_rank |= rank[jj] == rank[j];
        seen_node |= rank[jj] / a.ranks_per_node == node;
      }
      c[0] += 1;
      c[1] += !seen_rank;
      c[2] += !seen_node;
    }
  }
  for (int q = 0; q < 3; ++q) {
    int64_t v = c[q];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[q][warp] = v;
  }
  __syncthreads();
  if (tid < 3) {
    int64_t v = 0;
    for (int w = 0; w < kStatsThreads / 32; ++w) v += red[tid][w];
    a.stats[static_cast<int64_t>(src) * 4 + 1 + tid] = v;
  }
  if (tid == 3) a.stats[static_cast<int64_t>(src) * 4] = a.T;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route_stats(const moe_desc *desc, const int32_t *topk_idx, int32_t ranks_per_node,
                                      int64_t *stats, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (ranks_per_node < 1 || stats == nullptr || err == nullptr || (s.ntok > 0 && topk_idx == nullptr))
    return MOE_EINVAL;
  if (!aligned4(topk_idx) || (reinterpret_cast<uintptr_t>(stats) & 7u) != 0 || !aligned4(err)) return MOE_EINVAL;
  StatsArgs a{topk_idx, stats, err, s.T, s.E, s.k, s.L, ranks_per_node};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.R), 1, 1);
  cfg.blockDim = dim3(kStatsThreads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  if (cudaLaunchKernelEx(&cfg, route_stats_kernel, a) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

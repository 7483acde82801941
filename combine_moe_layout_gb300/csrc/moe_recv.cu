// Receive side of dispatch: wait for the count + 1 signals, then pack the
// filled slots into contiguous expert-major buffers.
//
// Perplexity, "Efficient and portable mixture-of-experts communication",
// section "Dispatch": the receiver first waits for every token count, then
// copies the payloads into contiguous buffers that feed the grouped GEMM of the
// experts, keeping (source rank, expert, token) for combine. "NVSHMEM and
// DeepEP: GPU-initiated communication", low-latency section: the receive step
// is a separate hook the caller runs when it wants the data, after a send that
// only issued its writes.
//
// Two kernels, chained by programmatic dependent launch:
//   region_scan_kernel  one CTA: a bounded wait on each region's flag, a check
//                       that flag - 1 == count <= max_m, and the exclusive scan
//                       of the counts in (expert, source rank) order.
//   compact_kernel      one warp per packed row p < R*T*k: binary search of the
//                       region holding p, then the row, its scales and its
//                       header copied with 16-byte loads and stores, and p
//                       recorded in tok_packed[src][t][j] (the forward map the
//                       packed combine gathers through; -1 for a choice with
//                       no slot, which that warp's index p also covers). The grid is
//                       the largest possible packed size, so the host needs no
//                       count and the call stays asynchronous.
#include "moe_common.cuh"

namespace moe {

constexpr int kScanThreads = 1024;
constexpr int kCompactWarps = 4;
constexpr int kCopyBatch = 8;  // 16-byte loads in flight per lane in the row copy

struct ScanArgs {
  const int32_t *counts;
  const uint64_t *flags;
  int32_t *region_offsets;
  int32_t *err;
  int64_t nreg;
  int max_m;
};

__global__ void __launch_bounds__(kScanThreads) region_scan_kernel(ScanArgs a) {
  __shared__ int64_t warp_sums[kScanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dependency_wait();
  const int64_t per = (a.nreg + kScanThreads - 1) / kScanThreads;
  const int64_t r0 = tid * per, r1 = r0 + per < a.nreg ? r0 + per : a.nreg;
  int64_t sum = 0;
  for (int64_t r = r0; r < r1; ++r) {
    int c = a.counts[r];
    const uint64_t f = wait_flag_nonzero(a.flags + r);
    if (f == 0) {
      latch_error(a.err, MOE_ETIMEOUT);
    } else if (f - 1 != static_cast<uint64_t>(c)) {
      latch_error(a.err, MOE_EINVAL);  // counts and flags of different steps
    }
    if (c < 0 || c > a.max_m) {
      latch_error(a.err, MOE_EOVERFLOW);
      c = c < 0 ? 0 : a.max_m;
    }
    sum += c;
  }
  // block-wide exclusive scan of the per-thread sums
  int64_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int64_t w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int64_t acc = incl - sum + (warp > 0 ? warp_sums[warp - 1] : 0);
  for (int64_t r = r0; r < r1; ++r) {
    a.region_offsets[r] = static_cast<int32_t>(acc);
    int c = a.counts[r];
    c = c < 0 ? 0 : (c > a.max_m ? a.max_m : c);
    acc += c;
  }
  if (tid == kScanThreads - 1) a.region_offsets[a.nreg] = static_cast<int32_t>(acc);
  grid_dependents_launch();
}

struct CompactArgs {
  const uint8_t *recv_x;
  const float *recv_scales;
  const int4 *recv_meta;
  const int32_t *tok_slot;
  const int32_t *region_offsets;
  uint8_t *packed_x;
  float *packed_scales;
  int4 *packed_meta;
  int32_t *tok_packed;
  int64_t nreg, npacked_max;
  int T, k, max_m, nsc;
  uint32_t row_bytes;
};

__global__ void __launch_bounds__(kCompactWarps * 32) compact_kernel(CompactArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t p = static_cast<int64_t>(blockIdx.x) * kCompactWarps + (threadIdx.x >> 5);
  grid_dependency_wait();
  // choice p (in [R][T][k] order) with no slot (masked, or rejected by layout)
  // has no packed row: its forward-map entry says so. Packed rows write only
  // the entries of choices that have a slot, so the two never meet.
  if (lane == 0 && p < a.npacked_max && a.tok_slot[p] < 0) a.tok_packed[p] = -1;
  if (p >= a.npacked_max || p >= a.region_offsets[a.nreg]) return;
  // the region r with offsets[r] <= p < offsets[r + 1]
  int64_t lo = 0, hi = a.nreg - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (a.region_offsets[mid] <= p)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int64_t pos = p - a.region_offsets[lo];
  if (pos < 0 || pos >= a.max_m) return;
  const int64_t slot = lo * a.max_m + pos;
  const uint4 *src = reinterpret_cast<const uint4 *>(a.recv_x + slot * a.row_bytes);
  uint4 *dst = reinterpret_cast<uint4 *>(a.packed_x + p * a.row_bytes);
  // kCopyBatch loads in flight per lane before their stores: one dependent
  // load -> store per 16 bytes would leave a warp with 512 bytes in flight,
  // too little to cover DRAM latency with the warps an SM holds
  const uint32_t nv = a.row_bytes / 16;
  uint32_t v = lane;
  for (; v + (kCopyBatch - 1) * 32 < nv; v += kCopyBatch * 32) {
    uint4 t[kCopyBatch];
#pragma unroll
    for (int b = 0; b < kCopyBatch; ++b) t[b] = __ldcs(src + v + b * 32);
#pragma unroll
    for (int b = 0; b < kCopyBatch; ++b) dst[v + b * 32] = t[b];
  }
  for (; v < nv; v += 32) dst[v] = __ldcs(src + v);
  for (int c = lane; c < a.nsc; c += 32) a.packed_scales[p * a.nsc + c] = a.recv_scales[slot * a.nsc + c];
  if (lane == 0) {
    // the header {src, t, e, j} also gives combine its forward map to the packed row
    const int4 m = a.recv_meta[slot];
    a.packed_meta[p] = m;
    if (m.y >= 0 && m.y < a.T && m.w >= 0 && m.w < a.k && m.x >= 0 && static_cast<int64_t>(m.x) * a.T * a.k < a.npacked_max)
      a.tok_packed[(static_cast<int64_t>(m.x) * a.T + m.y) * a.k + m.w] = static_cast<int32_t>(p);
  }
}

moe_status launch_recv(const Sizes &s, const int32_t *counts, const uint64_t *flags, const void *recv_x,
                       const float *recv_scales, const int32_t *recv_meta, const int32_t *tok_slot,
                       int32_t *region_offsets, void *packed_x, float *packed_scales, int32_t *packed_meta,
                       int32_t *tok_packed, int32_t *err, cudaStream_t stream) {
  ScanArgs sa{counts, flags, region_offsets, err, static_cast<int64_t>(s.E) * s.R, s.max_m};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kScanThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  if (cudaLaunchKernelEx(&cfg, region_scan_kernel, sa) != cudaSuccess) return MOE_ECUDA;
  if (launch_status() != MOE_OK) return MOE_ECUDA;
  const int64_t npacked = s.ntok * s.k;
  if (npacked == 0) return MOE_OK;
  CompactArgs ca{static_cast<const uint8_t *>(recv_x), recv_scales, reinterpret_cast<const int4 *>(recv_meta),
                 tok_slot, region_offsets, static_cast<uint8_t *>(packed_x), packed_scales,
                 reinterpret_cast<int4 *>(packed_meta), tok_packed, sa.nreg, npacked, s.T, s.k, s.max_m, s.nsc,
                 static_cast<uint32_t>(s.row_bytes)};
  const int64_t blocks = (npacked + kCompactWarps - 1) / kCompactWarps;
  if (blocks > 0x7fffffffll) return MOE_EINVAL;
  cudaLaunchConfig_t cc = {};
  cc.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cc.blockDim = dim3(kCompactWarps * 32, 1, 1);
  cc.stream = stream;
  cudaLaunchAttribute attr2[1];
  use_pdl(cc, attr2);
  if (cudaLaunchKernelEx(&cc, compact_kernel, ca) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch_recv(const moe_desc *desc, const int32_t *counts, const uint64_t *flags,
                                        const void *recv_x, const float *recv_scales, const int32_t *recv_meta,
                                        const int32_t *tok_slot, int32_t *region_offsets, void *packed_x,
                                        float *packed_scales, int32_t *packed_meta, int32_t *tok_packed,
                                        int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (counts == nullptr || flags == nullptr || region_offsets == nullptr || err == nullptr) return MOE_EINVAL;
  if (s.ntok > 0 && (recv_x == nullptr || recv_meta == nullptr || tok_slot == nullptr || packed_x == nullptr ||
                     packed_meta == nullptr || tok_packed == nullptr))
    return MOE_EINVAL;
  if (s.nsc > 0 && s.ntok > 0 && (recv_scales == nullptr || packed_scales == nullptr)) return MOE_EINVAL;
  if (!aligned16(recv_x) || !aligned16(packed_x) || !aligned16(recv_meta) || !aligned16(packed_meta) ||
      !aligned4(counts) || !aligned4(region_offsets) || !aligned4(err) || !aligned4(recv_scales) ||
      !aligned4(packed_scales) || !aligned4(tok_packed) || !aligned4(tok_slot) ||
      (reinterpret_cast<uintptr_t>(flags) & 7u) != 0)
    return MOE_EINVAL;
  return launch_recv(s, counts, flags, recv_x, recv_scales, recv_meta, tok_slot, region_offsets, packed_x,
                     packed_scales, packed_meta, tok_packed, err, static_cast<cudaStream_t>(stream));
}

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
// One kernel, recv_kernel, for up to kRecvMaxRegions (expert, source) regions:
// every CTA computes the exclusive scan of the counts (clamped to max_m) in
// its shared memory, the CTAs share the bounded waits on the regions' flags
// (and the check flag - 1 == count <= max_m), CTA 0 writes region_offsets, and
// then one warp per packed row p < R*T*k finds p's region by binary search in
// shared memory and copies the row, its scales and its header with 16-byte
// loads and stores, recording p in tok_packed[src][t][j] (the forward map the
// packed combine gathers through; -1 for a choice with no slot, which that
// warp's index p also covers). The grid is the resident capacity and the rows
// are the largest possible packed size, so the host needs no count and the
// call stays asynchronous. With more regions, two kernels chained by
// programmatic dependent launch do the same: region_scan_kernel (one CTA: the
// waits, the checks, the scan) and compact_kernel (the rows).
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

__device__ __forceinline__ void copy_packed_row(const CompactArgs &a, int64_t p, int64_t slot, int lane);

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
  copy_packed_row(a, p, slot, lane);
}

constexpr int kRecvThreads = 256;
constexpr int kRecvWarps = kRecvThreads / 32;
constexpr int64_t kRecvMaxRegions = 8192;

struct RecvArgs {
  const int32_t *counts;
  const uint64_t *flags;
  int32_t *region_offsets;
  int32_t *err;
  CompactArgs c;
  int early;
};

// The copy of packed row p from slot `slot` by one warp, shared by both forms
// of the receive hook. The header and the first scales are loaded first; then
// each pass has every lane issue up to kCopyBatch 16-byte loads (the last pass
// of a row predicated, not a run of single dependent load -> store steps)
// before its stores.
__device__ __forceinline__ void copy_packed_row(const CompactArgs &a, int64_t p, int64_t slot, int lane) {
  const uint4 *src = reinterpret_cast<const uint4 *>(a.recv_x + slot * a.row_bytes);
  uint4 *dst = reinterpret_cast<uint4 *>(a.packed_x + p * a.row_bytes);
  const uint32_t nv = a.row_bytes / 16;
  int4 m = make_int4(0, 0, 0, 0);
  if (lane == 0) m = a.recv_meta[slot];
  float sc0 = 0.0f;
  if (lane < a.nsc) sc0 = a.recv_scales[slot * a.nsc + lane];
  for (uint32_t v = lane; v < nv; v += kCopyBatch * 32) {
    uint4 t[kCopyBatch];
#pragma unroll
    for (int b = 0; b < kCopyBatch; ++b)
      if (v + b * 32 < nv) t[b] = __ldcs(src + v + b * 32);
#pragma unroll
    for (int b = 0; b < kCopyBatch; ++b)
      if (v + b * 32 < nv) dst[v + b * 32] = t[b];
  }
  if (lane < a.nsc) a.packed_scales[p * a.nsc + lane] = sc0;
  for (int c = lane + 32; c < a.nsc; c += 32) a.packed_scales[p * a.nsc + c] = a.recv_scales[slot * a.nsc + c];
  if (lane == 0) {
    // the header {src, t, e, j} also gives combine its forward map to the packed row
    a.packed_meta[p] = m;
    if (m.y >= 0 && m.y < a.T && m.w >= 0 && m.w < a.k && m.x >= 0 &&
        static_cast<int64_t>(m.x) * a.T * a.k < a.npacked_max)
      a.tok_packed[(static_cast<int64_t>(m.x) * a.T + m.y) * a.k + m.w] = static_cast<int32_t>(p);
  }
}

__global__ void __launch_bounds__(kRecvThreads) recv_kernel(RecvArgs a) {
  extern __shared__ int32_t s_off[];  // [nreg + 1]: exclusive scan of the clamped counts, then the total
  __shared__ int32_t warp_sums[kRecvWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nreg = static_cast<int>(a.c.nreg);
  grid_dependency_wait();
  if (a.early) grid_dependents_launch();

  // this CTA's share of the regions: bounded wait on the count + 1 flag, checks
  for (int r = blockIdx.x * kRecvThreads + tid; r < nreg; r += gridDim.x * kRecvThreads) {
    const int c = a.counts[r];
    const uint64_t f = wait_flag_nonzero(a.flags + r);
    if (f == 0)
      latch_error(a.err, MOE_ETIMEOUT);
    else if (f - 1 != static_cast<uint64_t>(c))
      latch_error(a.err, MOE_EINVAL);  // counts and flags of different steps
    if (c < 0 || c > a.c.max_m) latch_error(a.err, MOE_EOVERFLOW);
  }

  // exclusive scan of the clamped counts: thread tid owns regions [r0, r1)
  const int per = (nreg + kRecvThreads - 1) / kRecvThreads;
  const int r0 = min(tid * per, nreg), r1 = min(r0 + per, nreg);
  int sum = 0;
  for (int r = r0; r < r1; ++r) sum += min(max(a.counts[r], 0), a.c.max_m);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_sums[w];
  int acc = before + incl - sum;
  for (int r = r0; r < r1; ++r) {
    s_off[r] = acc;
    acc += min(max(a.counts[r], 0), a.c.max_m);
  }
  if (tid == kRecvThreads - 1) s_off[nreg] = acc;
  __syncthreads();
  if (blockIdx.x == 0)
    for (int r = tid; r <= nreg; r += kRecvThreads) a.region_offsets[r] = s_off[r];
  const int64_t total = s_off[nreg];

  // the rows: one warp per packed row
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * kRecvWarps + warp; p < a.c.npacked_max;
       p += static_cast<int64_t>(gridDim.x) * kRecvWarps) {
    // choice p with no slot (masked, or rejected by layout) has no packed row
    if (lane == 0 && a.c.tok_slot[p] < 0) a.c.tok_packed[p] = -1;
    if (p >= total) continue;
    int lo = 0, hi = nreg - 1;  // the region with s_off[lo] <= p < s_off[lo + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (s_off[mid] <= p)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int64_t pos = p - s_off[lo];
    if (pos < 0 || pos >= a.c.max_m) continue;
    copy_packed_row(a.c, p, static_cast<int64_t>(lo) * a.c.max_m + pos, lane);
  }
}

moe_status launch_recv(const Sizes &s, const int32_t *counts, const uint64_t *flags, const void *recv_x,
                       const float *recv_scales, const int32_t *recv_meta, const int32_t *tok_slot,
                       int32_t *region_offsets, void *packed_x, float *packed_scales, int32_t *packed_meta,
                       int32_t *tok_packed, int32_t *err, cudaStream_t stream) {
  const int64_t nreg = static_cast<int64_t>(s.E) * s.R;
  const int64_t npacked = s.ntok * s.k;
  CompactArgs ca{static_cast<const uint8_t *>(recv_x), recv_scales, reinterpret_cast<const int4 *>(recv_meta),
                 tok_slot, region_offsets, static_cast<uint8_t *>(packed_x), packed_scales,
                 reinterpret_cast<int4 *>(packed_meta), tok_packed, nreg, npacked, s.T, s.k, s.max_m, s.nsc,
                 static_cast<uint32_t>(s.row_bytes)};
  if (nreg <= kRecvMaxRegions) {
    RecvArgs ra{counts, flags, region_offsets, err, ca, early_trigger(s.ntok)};
    const size_t smem = static_cast<size_t>(nreg + 1) * sizeof(int32_t);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(recv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
      return MOE_ECUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, recv_kernel, kRecvThreads, smem) != cudaSuccess)
      return MOE_ECUDA;
    if (per_sm < 1) return MOE_EINVAL;
    int64_t grid = static_cast<int64_t>(sm_count()) * per_sm;
    const int64_t need = (npacked + kRecvWarps - 1) / kRecvWarps;
    if (grid > need) grid = need > 0 ? need : 1;
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    rc.blockDim = dim3(kRecvThreads, 1, 1);
    rc.dynamicSmemBytes = smem;
    rc.stream = stream;
    cudaLaunchAttribute ra_attr[1];
    use_pdl(rc, ra_attr);
    if (cudaLaunchKernelEx(&rc, recv_kernel, ra) != cudaSuccess) return MOE_ECUDA;
    return launch_status();
  }
  ScanArgs sa{counts, flags, region_offsets, err, nreg, s.max_m};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kScanThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  if (cudaLaunchKernelEx(&cfg, region_scan_kernel, sa) != cudaSuccess) return MOE_ECUDA;
  if (launch_status() != MOE_OK) return MOE_ECUDA;
  if (npacked == 0) return MOE_OK;
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

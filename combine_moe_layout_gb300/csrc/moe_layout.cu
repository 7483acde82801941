// Layout (K1): per-(expert, source rank) counts, count+1 flags and the fixed
// slot of every (source rank, token, choice).
//
// Perplexity, "Efficient and portable mixture-of-experts communication",
// section "Dispatch": the sender counts how many of its tokens each destination
// expert receives and signals count + 1, so that the change from zero means
// "count arrived". "NVSHMEM and DeepEP: GPU-initiated communication",
// low-latency section: every source rank owns max_m slots per local expert of
// each receiver, so a sender finds its slot with no exchange and no host sync.
//
// Design: one CTA per (chunk of 128 tokens, source rank). Positions are the
// token-order rank of an entry among the entries of its (expert, source) pair,
// so the result is deterministic and needs no grid-wide step:
//   1. the CTA histograms the entries of the source rank's earlier chunks
//      (warp-aggregated with match.any; L2-resident reads), giving the base of
//      every expert;
//   2. it builds a 128-bit membership bitmap per expert for its own chunk
//      (a repeated expert in one token shows up as a bit already set);
//   3. pos = base + popcount of the bitmap below the token;
//   4. the last chunk of a source rank owns the totals and writes counts and
//      flags = count + 1. Consumers are later kernels in stream order, which
//      see them once this grid completes (griddepcontrol.wait under
//      programmatic dependent launch), so plain stores suffice: a release fence
//      per flag would only lengthen this latency-bound kernel.
//
// Large batches (more than 128 tokens per rank) use a thread-block cluster per
// source rank instead: CTA r of the cluster owns tokens [r*TPC, (r+1)*TPC),
// builds the bitmaps of its slice, publishes its per-expert counts in its own
// shared memory, and after a cluster barrier sums the counts of CTAs 0..r-1
// through distributed shared memory to get its bases. Every entry is counted
// once, with no global scratch and no grid-wide step; the last CTA of the
// cluster writes the totals.
#include <cooperative_groups.h>

#include "moe_common.cuh"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kLayoutChunk = 128;
constexpr int kLayoutWords = kLayoutChunk / 32;
constexpr int kLayoutThreads = 512;
constexpr int kLayoutMaxExperts = 8192;

struct LayoutArgs {
  const int32_t *topk_idx;
  int32_t *counts;
  SlotParts parts;  // only the flags are written
  int32_t *tok_slot;
  int32_t *err;
  int R, T, E, k, max_m, early;
};

__global__ void __launch_bounds__(kLayoutThreads) layout_kernel(LayoutArgs a) {
  extern __shared__ uint32_t lsm[];
  int32_t *hist = reinterpret_cast<int32_t *>(lsm);
  uint32_t *bits = lsm + a.E;
  const int src = blockIdx.y;
  const int chunk = blockIdx.x;
  const int t0 = chunk * kLayoutChunk;
  const int tn = max(0, min(kLayoutChunk, a.T - t0));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;

  grid_dependency_wait();
  if (a.early) grid_dependents_launch();  // dispatch may start loading its rows meanwhile
  for (int i = tid; i < a.E * (1 + kLayoutWords); i += blockDim.x) lsm[i] = 0;
  __syncthreads();

  const int32_t *idx = a.topk_idx + static_cast<int64_t>(src) * a.T * a.k;

  // 1. base of every expert: entries of this source rank's earlier tokens
  const int n_prev = t0 * a.k;
  for (int base = warp * 32; base < n_prev; base += nwarps * 32) {
    const int i = base + lane;
    const int e = i < n_prev ? __ldg(idx + i) : -1;
    const bool ok = e >= 0 && e < a.E;
    const unsigned active = __ballot_sync(0xffffffffu, ok);
    if (ok) {
      const unsigned peers = __match_any_sync(active, e);
      if (lane == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
    }
  }

  // 2. membership bitmap of this chunk, per expert
  const int n_own = tn * a.k;
  const int32_t *own = idx + static_cast<int64_t>(t0) * a.k;
  for (int i = tid; i < n_own; i += blockDim.x) {
    const int e = __ldg(own + i);
    if (e < 0 || e >= a.E) {
      if (e != kMaskedExpert) latch_error(a.err, MOE_EINVAL);  // a masked choice is skipped silently
      continue;
    }
    const int tl = i / a.k;
    const uint32_t bit = 1u << (tl & 31);
    const uint32_t old = atomicOr(&bits[e * kLayoutWords + (tl >> 5)], bit);
    if (old & bit) latch_error(a.err, MOE_EINVAL);  // expert repeated within a token
  }
  __syncthreads();

  // 3. slot of every entry of this chunk
  int32_t *out = a.tok_slot + (static_cast<int64_t>(src) * a.T + t0) * a.k;
  for (int i = tid; i < n_own; i += blockDim.x) {
    const int e = __ldg(own + i);
    int32_t slot = -1;
    if (e >= 0 && e < a.E) {
      const int tl = i / a.k;
      const uint32_t *b = bits + e * kLayoutWords;
      int pos = hist[e];
      for (int w = 0; w < (tl >> 5); ++w) pos += __popc(b[w]);
      pos += __popc(b[tl >> 5] & ((1u << (tl & 31)) - 1u));
      if (pos < a.max_m)
        slot = static_cast<int32_t>((static_cast<int64_t>(e) * a.R + src) * a.max_m + pos);
      else
        latch_error(a.err, MOE_EOVERFLOW);
    }
    out[i] = slot;
  }

  // 4. totals: counts and count + 1 flags, published by the last chunk
  if (chunk == static_cast<int>(gridDim.x) - 1) {
    for (int e = tid; e < a.E; e += blockDim.x) {
      int c = hist[e];
#pragma unroll
      for (int w = 0; w < kLayoutWords; ++w) c += __popc(bits[e * kLayoutWords + w]);
      const int64_t r = static_cast<int64_t>(e) * a.R + src;
      a.counts[r] = c;
      *flag_ptr(a.parts, r) = static_cast<uint64_t>(c) + 1;
    }
  }
}

constexpr int kClusterMax = 8;             // portable cluster size
constexpr int kClusterThreads = 512;
constexpr int kClusterTokensPerCta = 512;
constexpr size_t kClusterMaxSmem = 200 * 1024;

__global__ void __launch_bounds__(kClusterThreads) layout_cluster_kernel(LayoutArgs a, int tpc, int words) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ uint32_t csm[];
  uint32_t *bits = csm;                                           // [E][words]
  int32_t *hist = reinterpret_cast<int32_t *>(csm + a.E * words);  // [E] counts of this slice
  int32_t *base = hist + a.E;                                     // [E] counts of the earlier slices
  const int r = static_cast<int>(cluster.block_rank());
  const int csize = static_cast<int>(cluster.num_blocks());
  const int src = blockIdx.y;
  const int t0 = r * tpc;
  const int tn = max(0, min(tpc, a.T - t0));
  const int tid = threadIdx.x;

  grid_dependency_wait();
  if (a.early) grid_dependents_launch();
  for (int i = tid; i < a.E * words; i += blockDim.x) bits[i] = 0;
  __syncthreads();

  const int32_t *own = a.topk_idx + (static_cast<int64_t>(src) * a.T + t0) * a.k;
  const int n_own = tn * a.k;
  for (int i = tid; i < n_own; i += blockDim.x) {
    const int e = __ldg(own + i);
    if (e < 0 || e >= a.E) {
      if (e != kMaskedExpert) latch_error(a.err, MOE_EINVAL);  // a masked choice is skipped silently
      continue;
    }
    const int tl = i / a.k;
    const uint32_t bit = 1u << (tl & 31);
    if (atomicOr(&bits[e * words + (tl >> 5)], bit) & bit) latch_error(a.err, MOE_EINVAL);
  }
  __syncthreads();
  for (int e = tid; e < a.E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < words; ++w) c += __popc(bits[e * words + w]);
    hist[e] = c;
  }
  cluster.sync();  // every slice's counts are visible to the whole cluster

  for (int e = tid; e < a.E; e += blockDim.x) {
    int b = 0;
    for (int q = 0; q < r; ++q) b += *cluster.map_shared_rank(hist + e, q);
    base[e] = b;
    if (r == csize - 1) {
      const int c = b + hist[e];
      const int64_t reg = static_cast<int64_t>(e) * a.R + src;
      a.counts[reg] = c;
      *flag_ptr(a.parts, reg) = static_cast<uint64_t>(c) + 1;
    }
  }
  __syncthreads();

  int32_t *out = a.tok_slot + (static_cast<int64_t>(src) * a.T + t0) * a.k;
  for (int i = tid; i < n_own; i += blockDim.x) {
    const int e = __ldg(own + i);
    int32_t slot = -1;
    if (e >= 0 && e < a.E) {
      const int tl = i / a.k;
      const uint32_t *b = bits + e * words;
      int pos = base[e];
      for (int w = 0; w < (tl >> 5); ++w) pos += __popc(b[w]);
      pos += __popc(b[tl >> 5] & ((1u << (tl & 31)) - 1u));
      if (pos < a.max_m)
        slot = static_cast<int32_t>((static_cast<int64_t>(e) * a.R + src) * a.max_m + pos);
      else
        latch_error(a.err, MOE_EOVERFLOW);
    }
    out[i] = slot;
  }
  cluster.sync();  // no CTA leaves while another may still read its counts
}

// Cluster shape for a batch, or false when the chunked kernel must be used.
static bool cluster_shape(const Sizes &s, int *csize, int *tpc, int *words, size_t *smem) {
  if (s.T <= kLayoutChunk) return false;
  int c = (s.T + kClusterTokensPerCta - 1) / kClusterTokensPerCta;
  if (c > kClusterMax) c = kClusterMax;
  if (c < 1) c = 1;
  int per = (s.T + c - 1) / c;
  per = (per + 31) / 32 * 32;
  *csize = c;
  *tpc = per;
  *words = per / 32;
  *smem = (static_cast<size_t>(s.E) * *words + 2 * static_cast<size_t>(s.E)) * sizeof(uint32_t);
  return *smem <= kClusterMaxSmem;
}

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

moe_status launch_layout(const Sizes &s, const int32_t *topk_idx, int32_t *counts, const SlotParts &parts,
                         int32_t *tok_slot, int32_t *err, cudaStream_t stream) {
  if (s.E > kLayoutMaxExperts) return MOE_EINVAL;
  LayoutArgs a{topk_idx, counts, parts, tok_slot, err, s.R, s.T, s.E, s.k, s.max_m, early_trigger(s.ntok)};
  int csize = 0, tpc = 0, words = 0;
  size_t csmem = 0;
  if (cluster_shape(s, &csize, &tpc, &words, &csmem)) {
    if (csmem > 48 * 1024 && cudaFuncSetAttribute(layout_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(csmem)) != cudaSuccess)
      return MOE_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize, s.R, 1);
    cfg.blockDim = dim3(kClusterThreads, 1, 1);
    cfg.dynamicSmemBytes = csmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = csize;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, layout_cluster_kernel, a, tpc, words) != cudaSuccess) return MOE_ECUDA;
    return launch_status();
  }
  const size_t smem = static_cast<size_t>(s.E) * (1 + kLayoutWords) * sizeof(uint32_t);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return MOE_ECUDA;
  const int chunks = s.T > 0 ? (s.T + kLayoutChunk - 1) / kLayoutChunk : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(chunks, s.R, 1);
  cfg.blockDim = dim3(kLayoutThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  if (cudaLaunchKernelEx(&cfg, layout_kernel, a) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_buffer_sizes(const moe_desc *desc, moe_sizes *out) {
  Sizes s;
  const moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (out == nullptr) return MOE_EINVAL;
  const size_t slots = static_cast<size_t>(s.nslots);
  out->recv_x = slots * static_cast<size_t>(s.row_bytes);
  out->recv_scales = slots * static_cast<size_t>(s.nsc) * sizeof(float);
  out->recv_meta = slots * 4 * sizeof(int32_t);
  out->counts = static_cast<size_t>(s.E) * s.R * sizeof(int32_t);
  out->flags = static_cast<size_t>(s.E) * s.R * sizeof(uint64_t);
  out->tok_slot = static_cast<size_t>(s.ntok) * s.k * sizeof(int32_t);
  out->expert_out = slots * static_cast<size_t>(s.H) * 2;
  return MOE_OK;
}

extern "C" moe_status moe_layout(const moe_desc *desc, const int32_t *topk_idx, int32_t *counts, uint64_t *flags,
                                 int32_t *tok_slot, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (counts == nullptr || flags == nullptr || err == nullptr) return MOE_EINVAL;
  if (s.ntok > 0 && (topk_idx == nullptr || tok_slot == nullptr)) return MOE_EINVAL;
  if (!aligned4(topk_idx) || !aligned4(counts) || !aligned4(tok_slot) || !aligned4(err) ||
      (reinterpret_cast<uintptr_t>(flags) & 7u) != 0)
    return MOE_EINVAL;
  return launch_layout(s, topk_idx, counts, single_part(s, nullptr, nullptr, nullptr, flags, nullptr), tok_slot, err,
                       static_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_reset(const moe_desc *desc, uint64_t *flags, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (flags == nullptr || err == nullptr) return MOE_EINVAL;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(flags, 0, static_cast<size_t>(s.E) * s.R * sizeof(uint64_t), cs) != cudaSuccess)
    return MOE_ECUDA;
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), cs) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

extern "C" moe_status moe_reset_parts(const moe_desc *desc, const moe_parts *parts, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  SlotParts p;
  st = parts_from(s, parts, false, false, &p);
  if (st != MOE_OK) return st;
  if (err == nullptr) return MOE_EINVAL;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  for (int g = 0; g < p.G; ++g)
    if (cudaMemsetAsync(p.flags[g], 0, static_cast<size_t>(p.regions_per_part) * sizeof(uint64_t), cs) != cudaSuccess)
      return MOE_ECUDA;
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), cs) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

extern "C" moe_status moe_get_error(int32_t *err, void *stream) {
  if (err == nullptr) return MOE_EINVAL;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof v, cudaMemcpyDeviceToHost, cs) != cudaSuccess) return MOE_ECUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return MOE_ECUDA;
  if (v != 0) {
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), cs) != cudaSuccess) return MOE_ECUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return MOE_ECUDA;
  }
  return static_cast<moe_status>(v);
}

extern "C" const char *moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument or routing";
    case MOE_EOVERFLOW: return "more tokens for an (expert, source rank) than max_m slots";
    case MOE_ETIMEOUT: return "bounded wait on a count+1 flag gave up";
    case MOE_ECUDA: return "CUDA runtime error";
    case MOE_ENOMEM: return "out of device memory";
    default: return "unknown status";
  }
}

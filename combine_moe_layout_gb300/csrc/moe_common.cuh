// Shared device and host helpers of libmoe_layout (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_layout.h"

namespace moe {

constexpr int kMaxTopk = 16;
constexpr int kMaxStages = 8;  // row stages of the dispatch kernels
constexpr int kScaleBlock = 128;  // elements per fp32 scale of an fp8 row
constexpr int kMaskedExpert = -1;  // a topk_idx entry naming no expert: skipped, no error

// Limits of the bounded waits, in nanoseconds of %globaltimer. A count+1 flag
// is published by an earlier kernel in stream order, so a zero flag means the
// layout step did not run: give up after 1 ms instead of hanging. A TMA
// completion that never arrives would mean a fault: give up after 200 ms,
// far longer than any copy takes.
constexpr uint64_t kFlagWaitNs = 1000000ull;
constexpr uint64_t kMbarWaitNs = 200000000ull;
constexpr unsigned kFlagSleepNs = 128;

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Error word: the first error a kernel finds wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void latch_error(int32_t *err, int32_t code) {
  if (err != nullptr && *reinterpret_cast<volatile int32_t *>(err) == 0) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// Flags: count + 1 signals, published with release and polled with acquire.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_release_u64(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t load_acquire_u64(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *flag != 0; returns the flag (0 after giving up).
__device__ __forceinline__ uint64_t wait_flag_nonzero(const uint64_t *flag) {
  uint64_t v = load_acquire_u64(flag);
  if (v != 0) return v;
  const uint64_t t0 = global_timer_ns();
  while (v == 0 && global_timer_ns() - t0 < kFlagWaitNs) {
    __nanosleep(kFlagSleepNs);
    v = load_acquire_u64(flag);
  }
  return v;
}

// ---------------------------------------------------------------------------
// mbarrier and bulk (non-tensor) TMA copies.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's generic-proxy shared memory accesses before later
// async-proxy (TMA) accesses to the same shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of an mbarrier; false after giving up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < kMbarWaitNs)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Shared -> global bulk copy tracked by bulk groups.
__device__ __forceinline__ void bulk_store(void *gmem_dst, const void *smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk group has completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Programmatic dependent launch: wait for the preceding kernel's results, and
// allow the next kernel to start its prologue.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Quantise-on-dispatch: bf16 blocks of 128 elements -> E4M3 + one fp32 scale.
// scale = amax / 448 (1 for an all-zero block); code = e4m3(x / scale), with
// IEEE fp32 division and the hardware's round-to-nearest-even, saturating
// conversion. Warp w of nwarps handles blocks w, w + nwarps, ...; each lane
// takes 4 consecutive elements. src, dst and sc are shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint16_t e4m3x2_rn_satfinite(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;  // lo in the low byte, hi in the high byte
}

// The block scale of a 128-element block and what the code helper below needs:
// s = amax / 448 (IEEE fp32; 1 for an all-zero block), r = 1/s rounded to
// nearest, and r scaled by 1 - 2^-20 and 1 + 2^-20. fast is false where 1/s
// could leave the normal range (s below 2^-125, or not finite).
struct BlockScale {
  float s, lo, hi;
  bool fast;
};

__device__ __forceinline__ BlockScale block_scale(float amax) {
  BlockScale b;
  b.s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  b.fast = b.s >= 0x1p-125f && b.s <= 0x1p+125f;
  const float r = __frcp_rn(b.s);
  b.lo = r * 0x1.ffffep-1f;  // 1 - 2^-20
  b.hi = r * 0x1.00001p+0f;  // 1 + 2^-20
  return b;
}

// The e4m3 codes of x0 / s and x1 / s: the IEEE fp32 quotients, converted with
// round to nearest even and saturation (low byte x0), in the common case
// without a division. With r = RN(1/s), three roundings of relative size at
// most 2^-24 separate x * RN(r (1 - 2^-20)) from x/s (1 - 2^-20), so it lies
// below x/s by a relative 2^-20 - 3 * 2^-24 or more, and x * RN(r (1 + 2^-20))
// lies above it by as much. The correctly rounded quotient is within 2^-24 of
// x/s, so the two products bracket it. The conversion is monotonic: when both
// products give the same codes, those are the quotient's. Where they differ
// (an e4m3 rounding boundary within about 2^-20 of the quotient, or a NaN) the
// quotients are computed by division. Products that fall to fp32 subnormals
// are below 2^-125 and code 0, as the quotient does.
__device__ __forceinline__ uint16_t e4m3x2_of_quotients(float x0, float x1, const BlockScale &b) {
  if (b.fast) {
    const uint16_t lo = e4m3x2_rn_satfinite(x0 * b.lo, x1 * b.lo);
    const uint16_t hi = e4m3x2_rn_satfinite(x0 * b.hi, x1 * b.hi);
    if (lo == hi) return lo;
  }
  return e4m3x2_rn_satfinite(__fdiv_rn(x0, b.s), __fdiv_rn(x1, b.s));
}

__device__ __forceinline__ void quantize_blocks(const uint16_t *src, uint8_t *dst, float *sc, int nblk, int warp,
                                                int nwarps, int lane) {
  for (int b = warp; b < nblk; b += nwarps) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(src + b * kScaleBlock + lane * 4);
    const float f0 = __uint_as_float(raw.x << 16), f1 = __uint_as_float(raw.x & 0xffff0000u);
    const float f2 = __uint_as_float(raw.y << 16), f3 = __uint_as_float(raw.y & 0xffff0000u);
    float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const BlockScale bs = block_scale(amax);
    const uint32_t q = static_cast<uint32_t>(e4m3x2_of_quotients(f0, f1, bs)) |
                       (static_cast<uint32_t>(e4m3x2_of_quotients(f2, f3, bs)) << 16);
    *reinterpret_cast<uint32_t *>(dst + b * kScaleBlock + lane * 4) = q;
    if (lane == 0) sc[b] = bs.s;
  }
}

// ---------------------------------------------------------------------------
// Slot partitions: the fixed-slot buffers (rows, scales, headers, count+1
// flags, expert outputs) split into G parts as G GPUs of an EP group would hold
// them. Part g holds the regions of ranks [g*R/G, (g+1)*R/G): global slots
// [g*P, (g+1)*P) at local slot s - g*P, with P = (R/G)*L*R*max_m, and regions
// likewise. Slot ids (tok_slot, headers) stay global. G = 1 is the single
// buffer; its address arithmetic takes a uniform branch and no division.
// ---------------------------------------------------------------------------
constexpr int kMaxParts = MOE_MAX_PARTS;

struct SlotParts {
  int G;
  int32_t slots_per_part;    // P
  int32_t regions_per_part;  // P / max_m
  uint8_t *recv_x[kMaxParts];
  float *recv_scales[kMaxParts];
  int4 *recv_meta[kMaxParts];
  uint64_t *flags[kMaxParts];
  uint16_t *y[kMaxParts];  // expert outputs (bf16 rows of H)
};

// Part and local index of a global slot (or region, with per = regions_per_part).
// Slot ids fit in 32 bits (the desc check bounds E*R*max_m), so 32-bit division.
__device__ __forceinline__ int part_split(int G, int32_t per, int64_t id, int64_t *local) {
  if (G == 1) {
    *local = id;
    return 0;
  }
  const uint32_t u = static_cast<uint32_t>(id);
  const uint32_t g = u / static_cast<uint32_t>(per);
  *local = static_cast<int64_t>(u - g * static_cast<uint32_t>(per));
  return static_cast<int>(g);
}

// Local slot of a global slot, and its part in *g.
__device__ __forceinline__ int64_t slot_local(const SlotParts &p, int64_t slot, int *g) {
  int64_t l;
  *g = part_split(p.G, p.slots_per_part, slot, &l);
  return l;
}

__device__ __forceinline__ uint64_t *flag_ptr(const SlotParts &p, int64_t region) {
  int64_t l;
  const int g = part_split(p.G, p.regions_per_part, region, &l);
  return p.flags[g] + l;
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
struct Sizes {
  int R, T, H, E, k, max_m, dtype, L;
  int64_t nslots;     // E * R * max_m
  int64_t ntok;       // R * T
  int64_t row_bytes;     // bytes of a dispatched row: 2H (bf16) or H (fp8, bf16-to-fp8)
  int64_t in_row_bytes;  // bytes of a caller's input row: H (fp8) or 2H (bf16, bf16-to-fp8)
  int nsc;               // scales per dispatched row (H/128, 0 for bf16)
  bool quant;            // bf16 input rows quantised to fp8 on dispatch
};

// Independent restatement of the desc rules (see moe_layout.h).
inline moe_status check_desc(const moe_desc *d, Sizes *s) {
  if (d == nullptr) return MOE_EINVAL;
  const int R = d->num_ranks, T = d->tokens_per_rank, H = d->hidden, E = d->num_experts, k = d->topk,
            M = d->max_m;
  if (R < 1 || T < 0 || H < 1 || E < 1 || k < 1 || M < 1) return MOE_EINVAL;
  if (E % R != 0 || k > E || k > kMaxTopk || T > M) return MOE_EINVAL;
  if (d->dtype == MOE_FP8_E4M3 || d->dtype == MOE_BF16_TO_FP8) {
    if (H % kScaleBlock != 0) return MOE_EINVAL;
  } else if (d->dtype == MOE_BF16) {
    if (H % 8 != 0) return MOE_EINVAL;
  } else {
    return MOE_EINVAL;
  }
  if (d->num_sms < 0) return MOE_EINVAL;
  if (static_cast<int64_t>(E) * R * M > INT32_MAX) return MOE_EINVAL;
  if (static_cast<int64_t>(R) * T * k > INT32_MAX) return MOE_EINVAL;
  if (s != nullptr) {
    s->R = R;
    s->T = T;
    s->H = H;
    s->E = E;
    s->k = k;
    s->max_m = M;
    s->dtype = d->dtype;
    s->L = E / R;
    s->nslots = static_cast<int64_t>(E) * R * M;
    s->ntok = static_cast<int64_t>(R) * T;
    s->row_bytes = d->dtype == MOE_BF16 ? 2 * static_cast<int64_t>(H) : H;
    s->in_row_bytes = d->dtype == MOE_FP8_E4M3 ? H : 2 * static_cast<int64_t>(H);
    s->nsc = d->dtype == MOE_BF16 ? 0 : H / kScaleBlock;
    s->quant = d->dtype == MOE_BF16_TO_FP8;
  }
  return MOE_OK;
}

inline bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline moe_status launch_status() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ECUDA; }

// SM count of the current device (queried once per device).
int sm_count();

// Launch with programmatic dependent launch (MOE_PDL=1): the kernel may be
// scheduled while the previous kernel in the stream finishes and waits for its
// results with griddepcontrol.wait.
#ifndef MOE_PDL
#define MOE_PDL 1
#endif
inline void use_pdl(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&attr)[1]) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

// Small batches let the next kernel launch as soon as this one has passed its
// own dependency wait (hiding the next launch behind this kernel); large ones
// do not, because the next kernel's CTAs would then sit on the SMs for the
// whole of a long kernel and slow it down.
#ifndef MOE_EARLY_TRIGGER_TOKENS
#define MOE_EARLY_TRIGGER_TOKENS 2048
#endif
inline int early_trigger(int64_t ntok) { return ntok <= MOE_EARLY_TRIGGER_TOKENS ? 1 : 0; }

// Units issued but not yet consumed when a pipelined loop aborts at unit i:
// the prologue issued units [0, S), and iteration u >= 1 refilled unit u-1+S,
// so the loads of units [i, end) may still be in flight.
__host__ __device__ inline int64_t inflight_end(int64_t i, int64_t S, int64_t n) {
  const int64_t end = i == 0 ? S : i - 1 + S;
  return end < n ? end : n;
}

// One buffer of each kind: the parts of a single-device step.
inline SlotParts single_part(const Sizes &s, void *recv_x, float *recv_scales, int32_t *recv_meta, uint64_t *flags,
                             const void *y) {
  SlotParts p{};
  p.G = 1;
  p.slots_per_part = static_cast<int32_t>(s.nslots);
  p.regions_per_part = s.E * s.R;
  p.recv_x[0] = static_cast<uint8_t *>(recv_x);
  p.recv_scales[0] = recv_scales;
  p.recv_meta[0] = reinterpret_cast<int4 *>(recv_meta);
  p.flags[0] = flags;
  p.y[0] = static_cast<uint16_t *>(const_cast<void *>(y));
  return p;
}

// The internal part table of a caller's moe_parts, checked: G divides R and is
// at most kMaxParts; the buffers each use are present and aligned (recv: rows,
// scales, headers and flags; y: expert outputs; flags are always needed).
inline moe_status parts_from(const Sizes &s, const moe_parts *p, bool need_recv, bool need_y, SlotParts *out) {
  if (p == nullptr) return MOE_EINVAL;
  const int G = p->num_parts;
  if (G < 1 || G > kMaxParts || s.R % G != 0) return MOE_EINVAL;
  SlotParts q{};
  q.G = G;
  q.slots_per_part = static_cast<int32_t>(s.nslots / G);
  q.regions_per_part = s.E * s.R / G;
  for (int g = 0; g < G; ++g) {
    if (p->flags[g] == nullptr || (reinterpret_cast<uintptr_t>(p->flags[g]) & 7u) != 0) return MOE_EINVAL;
    if (need_recv) {
      if (p->recv_x[g] == nullptr || p->recv_meta[g] == nullptr || !aligned16(p->recv_x[g]) ||
          !aligned16(p->recv_meta[g]))
        return MOE_EINVAL;
      if (s.nsc > 0 && (p->recv_scales[g] == nullptr || !aligned4(p->recv_scales[g]))) return MOE_EINVAL;
    }
    if (need_y && (p->expert_out[g] == nullptr || !aligned16(p->expert_out[g]))) return MOE_EINVAL;
    q.recv_x[g] = static_cast<uint8_t *>(p->recv_x[g]);
    q.recv_scales[g] = p->recv_scales[g];
    q.recv_meta[g] = reinterpret_cast<int4 *>(p->recv_meta[g]);
    q.flags[g] = p->flags[g];
    q.y[g] = static_cast<uint16_t *>(p->expert_out[g]);
  }
  *out = q;
  return MOE_OK;
}

moe_status launch_layout(const Sizes &s, const int32_t *topk_idx, int32_t *counts, const SlotParts &parts,
                         int32_t *tok_slot, int32_t *err, cudaStream_t stream);
moe_status launch_dispatch(const Sizes &s, const void *x, const float *x_scales, const int32_t *tok_slot,
                           const SlotParts &parts, int32_t *err, int num_sms, cudaStream_t stream);
moe_status launch_layout_dispatch(const Sizes &s, const int32_t *topk_idx, const void *x, const float *x_scales,
                                  int32_t *counts, int32_t *tok_slot, const SlotParts &parts, int32_t *err,
                                  int num_sms, cudaStream_t stream);
moe_status launch_combine(const Sizes &s, const SlotParts &parts, int64_t y_rows, const float *weights,
                          const int32_t *tok_slot, uint16_t *out, int32_t *err, cudaStream_t stream);

}  // namespace moe

// The expert stage (linear 1 with SwiGLU, then linear 2) as one call that
// allocates nothing: the intermediate h lives in a file-scope device array of
// fixed size instead of a caller buffer. The pages have no counterpart of this
// call; it serves callers that may not allocate device memory (for example
// inside a region captured into a CUDA graph with a fixed memory plan).
//
// The scratch is shared by every call on a device: two calls whose work
// overlaps in time (different streams, or graphs replayed concurrently) race on
// it. Rows of the scratch that a call does not write are read only into output
// rows that are never stored (rows past an expert's end), so it is not cleared.
#include "moe_common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // h of at most R*T*k x I bf16 = 32 MiB

static __device__ __align__(256) uint8_t g_expert_h_scratch[kScratchBytes];

// Device address of the scratch in the current context. In host code the
// array's name is only a stand-in, so the address is asked of the runtime on
// every call: the lookup is a host-side table read once the library's module
// is loaded in the context, and no address outlives a context (a cached one
// could, after cudaDeviceReset or with a non-primary context). The first call
// in a context loads the module: make it before any stream capture.
void *scratch_address() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_expert_h_scratch) != cudaSuccess) return nullptr;
  return p;
}

}  // namespace

extern "C" moe_status moe_expert_mlp_noalloc(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                             const void *packed_x, const void *w_gate, const void *w_up,
                                             const void *w_down, void *packed_y, int32_t *err, void *stream) {
  moe::Sizes s;
  const moe_status st = moe::check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (inter < 1) return MOE_EINVAL;
  const int64_t rows = s.ntok * s.k;
  if (static_cast<uint64_t>(rows) * static_cast<uint64_t>(inter) * 2u > kScratchBytes) return MOE_ENOMEM;
  void *h = scratch_address();
  if (h == nullptr) return MOE_ECUDA;
  const moe_status a = moe_expert_gate_up(desc, inter, region_offsets, packed_x, w_gate, w_up, h, err, stream);
  if (a != MOE_OK) return a;
  return moe_expert_down(desc, inter, region_offsets, h, w_down, packed_y, err, stream);
}

// The fp8 expert stage in one call that allocates nothing: h (e4m3, R*T*k x I
// bytes) at the start of the same scratch and its 128-element scales after it,
// at the next 256-byte boundary. The same race rule applies.
extern "C" moe_status moe_expert_mlp_noalloc_fp8(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                                 const void *packed_x, const float *packed_scales, const void *w_gate,
                                                 const float *w_gate_scales, const void *w_up,
                                                 const float *w_up_scales, const void *w_down,
                                                 const float *w_down_scales, void *packed_y, int32_t *err,
                                                 void *stream) {
  moe::Sizes s;
  const moe_status st = moe::check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (inter < 128 || inter % 128 != 0) return MOE_EINVAL;
  const uint64_t rows = static_cast<uint64_t>(s.ntok) * static_cast<uint64_t>(s.k);
  const uint64_t h_bytes = (rows * static_cast<uint64_t>(inter) + 255u) & ~uint64_t(255);
  const uint64_t sc_bytes = rows * static_cast<uint64_t>(inter / 128) * 4u;
  if (h_bytes + sc_bytes > kScratchBytes) return MOE_ENOMEM;
  uint8_t *h = static_cast<uint8_t *>(scratch_address());
  if (h == nullptr) return MOE_ECUDA;
  float *h_scales = reinterpret_cast<float *>(h + h_bytes);
  const moe_status a = moe_expert_gate_up_fp8(desc, inter, region_offsets, packed_x, packed_scales, w_gate,
                                              w_gate_scales, w_up, w_up_scales, h, h_scales, err, stream);
  if (a != MOE_OK) return a;
  return moe_expert_down_fp8(desc, inter, region_offsets, h, h_scales, w_down, w_down_scales, packed_y, err, stream);
}

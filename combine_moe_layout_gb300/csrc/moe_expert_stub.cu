// Synthetic experts for fp8 steps (not part of the pages' method; a stand-in
// for the expert MLPs that run between dispatch and combine, used by the tests
// and the benchmark).
//
// For every filled slot (pos < counts[region]) of expert e:
//   y[h] = bf16_rne( e4m3(q[h]) * scale[h / 128] * (1 + e/256) ).
// The product of a 4-bit e4m3 significand, a 24-bit fp32 scale and a 9-bit
// factor is exact in fp64, so y is that exact value rounded once to bf16.
#include "moe_common.cuh"

namespace moe {

constexpr int kStubThreads = 256;
constexpr int kStubSlotsPerRegionBlock = 8;

struct StubArgs {
  SlotParts parts;  // the rows and scales read, the expert outputs y written, per part
  const int32_t *counts;
  int32_t *err;
  int R, H, max_m, nsc;
};

// FP8 E4M3 ("e4m3fn") code -> exact double: sign, 4 exponent bits (bias 7),
// 3 mantissa bits; exponent 0 is subnormal (M * 2^-9); S.1111.111 is NaN.
__device__ __forceinline__ double e4m3_to_double(uint32_t b) {
  const uint32_t ex = (b >> 3) & 15u, m = b & 7u;
  double v;
  if (ex == 15u && m == 7u)
    v = __longlong_as_double(0x7ff8000000000000ll);
  else if (ex == 0u)
    v = static_cast<double>(m) * 0x1p-9;
  else
    v = __longlong_as_double(static_cast<long long>(((uint64_t)(ex - 7u + 1023u) << 52) | ((uint64_t)m << 49)));
  return (b & 0x80u) ? -v : v;
}

// Round a finite double to the nearest bfloat16 (ties to even), as bits.
// bfloat16 keeps 7 fraction bits in binary32's exponent range: for doubles of
// magnitude >= 2^-126 drop the low 45 fraction bits with round-half-even on the
// bit pattern (a carry into the exponent is the correct next binade); below
// 2^-126 the spacing is fixed at 2^-133.
__device__ __forceinline__ uint16_t bf16_rne_from_double(double v) {
  const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(v));
  const uint16_t sign = static_cast<uint16_t>((bits >> 48) & 0x8000u);
  uint64_t mag = bits & 0x7fffffffffffffffull;
  if (mag > 0x7ff0000000000000ull) return 0x7fc0;  // NaN
  double r;
  if (mag >= 0x3810000000000000ull) {  // |v| >= 2^-126
    mag += 0x00000fffffffffffull + ((mag >> 45) & 1u);
    mag &= ~0x00001fffffffffffull;
    r = __longlong_as_double(static_cast<long long>(mag));
    if (r >= 0x1p128) return static_cast<uint16_t>(sign | 0x7f80u);
  } else {
    r = rint(__longlong_as_double(static_cast<long long>(mag)) * 0x1p133) * 0x1p-133;
  }
  const float f = static_cast<float>(r);  // exact: at most 8 significant bits
  return static_cast<uint16_t>(sign | (__float_as_uint(f) >> 16));
}

__global__ void __launch_bounds__(kStubThreads) expert_stub_kernel(StubArgs a) {
  const int64_t region = blockIdx.x;
  int count = a.counts[region];
  if (count > a.max_m) {
    latch_error(a.err, MOE_EOVERFLOW);
    count = a.max_m;
  }
  const int e = static_cast<int>(region / a.R);
  const double c = 1.0 + static_cast<double>(e) / 256.0;
  int64_t lr;  // the region within its part
  const int g = part_split(a.parts.G, a.parts.regions_per_part, region, &lr);
  for (int pos = blockIdx.y; pos < count; pos += gridDim.y) {
    const int64_t s = lr * a.max_m + pos;
    const uint8_t *q = a.parts.recv_x[g] + s * a.H;
    const float *sc = a.parts.recv_scales[g] + s * a.nsc;
    uint16_t *y = a.parts.y[g] + s * a.H;
    for (int h = threadIdx.x * 8; h < a.H; h += kStubThreads * 8) {
      const uint2 packed = *reinterpret_cast<const uint2 *>(q + h);
      const double scale = static_cast<double>(sc[h / kScaleBlock]);
      uint32_t out[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t word = i < 2 ? packed.x : packed.y;
        const uint32_t b0 = (word >> (16 * (i & 1))) & 0xffu, b1 = (word >> (16 * (i & 1) + 8)) & 0xffu;
        const uint16_t y0 = bf16_rne_from_double(e4m3_to_double(b0) * scale * c);
        const uint16_t y1 = bf16_rne_from_double(e4m3_to_double(b1) * scale * c);
        out[i] = static_cast<uint32_t>(y0) | (static_cast<uint32_t>(y1) << 16);
      }
      *reinterpret_cast<uint4 *>(y + h) = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
}

}  // namespace moe

using namespace moe;

static moe_status launch_stub(const Sizes &s, const SlotParts &parts, const int32_t *counts, int32_t *err,
                              cudaStream_t stream) {
  StubArgs a{parts, counts, err, s.R, s.H, s.max_m, s.nsc};
  const int per_region = s.max_m < kStubSlotsPerRegionBlock ? s.max_m : kStubSlotsPerRegionBlock;
  dim3 grid(static_cast<unsigned>(s.E) * s.R, per_region, 1);
  expert_stub_kernel<<<grid, kStubThreads, 0, stream>>>(a);
  return launch_status();
}

extern "C" moe_status moe_expert_stub(const moe_desc *desc, const void *recv_x, const float *recv_scales,
                                      const int32_t *counts, uint16_t *expert_out, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (s.dtype == MOE_BF16) return MOE_EINVAL;
  if (recv_x == nullptr || recv_scales == nullptr || counts == nullptr || expert_out == nullptr || err == nullptr)
    return MOE_EINVAL;
  if (!aligned16(recv_x) || !aligned16(expert_out) || !aligned4(recv_scales) || !aligned4(counts))
    return MOE_EINVAL;
  SlotParts p = single_part(s, const_cast<void *>(recv_x), const_cast<float *>(recv_scales), nullptr, nullptr,
                            expert_out);
  return launch_stub(s, p, counts, err, static_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_expert_stub_parts(const moe_desc *desc, const moe_parts *parts, const int32_t *counts,
                                            int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (s.dtype == MOE_BF16) return MOE_EINVAL;
  SlotParts p;
  st = parts_from(s, parts, true, true, &p);
  if (st != MOE_OK) return st;
  if (counts == nullptr || err == nullptr || !aligned4(counts)) return MOE_EINVAL;
  return launch_stub(s, p, counts, err, static_cast<cudaStream_t>(stream));
}

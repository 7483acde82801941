// Dispatch (K2): copy every token row, with its fp32 block scales and a
// 16-byte header, into its k fixed slots.
//
// Perplexity, "Efficient and portable mixture-of-experts communication",
// section "Dispatch": activations, scales and the token's index on its own rank
// are packed and sent to each chosen expert; the receiver keeps (source rank,
// expert, token) for combine. "NVSHMEM and DeepEP: GPU-initiated
// communication": FP8 rows with one fp32 scale per 128 elements, written into
// the receiver's fixed slots. On one GPU a "put" into a peer's slot is a store
// into that rank's partition of the one allocation.
//
// Design: a work unit is (row, piece of at most 16 KiB). Each CTA is one warp
// and owns units blockIdx.x, blockIdx.x + gridDim.x, ... Lane 0 streams the
// unit bytes global -> shared with bulk TMA loads (S stages, one mbarrier
// each), and writes each staged piece to its k slots with bulk TMA stores
// (shared -> global, tracked by bulk groups); a stage is refilled once its
// stores have finished reading it. While a load is in flight, the other lanes
// read the unit's k slot ids, wait (bounded) on the count+1 flags of the
// destination regions, and write the headers and scales with plain stores.
// The grid is sized to the resident CTA count, so every load of a small batch
// is issued at once.
#include "moe_common.cuh"

namespace moe {

constexpr uint32_t kPieceMax = 16384;       // bytes staged per unit
constexpr uint32_t kStageBudget = 32768;    // shared bytes of staging per CTA

struct DispatchArgs {
  const uint8_t *x;
  const float *x_scales;
  const int32_t *tok_slot;
  SlotParts parts;  // rows, scales, headers and count + 1 flags of the receive side
  int32_t *err;
  int R, T, k, max_m, nsc, stages, pieces, early, quant;
  // row_bytes, piece_bytes: of the caller's input rows. Copy mode dispatches
  // them as they are; quant mode turns each 256-byte bf16 block of a piece into
  // 128 e4m3 bytes (the dispatched row has row_bytes / 2 bytes) and one scale.
  uint32_t row_bytes, piece_bytes;
  int64_t nslots, nunits;
};

__device__ __forceinline__ void issue_unit_load(const DispatchArgs &a, uint8_t *stage, uint64_t *bar, int64_t unit) {
  const int64_t row = unit / a.pieces;
  const uint32_t off = static_cast<uint32_t>(unit % a.pieces) * a.piece_bytes;
  const uint32_t bytes = min(a.piece_bytes, a.row_bytes - off);
  mbar_arrive_expect_tx(bar, bytes);
  bulk_load(stage, a.x + row * a.row_bytes + off, bytes, bar);
}

// Quant mode: shared memory holds S input stages, then S e4m3 stages of half
// their size, then S scale buffers of piece_bytes / 256 floats.
__device__ __forceinline__ uint8_t *qstage(const DispatchArgs &a, uint8_t *base, int s) {
  return base + static_cast<size_t>(a.stages) * a.piece_bytes + static_cast<size_t>(s) * (a.piece_bytes / 2);
}
__device__ __forceinline__ float *qscales(const DispatchArgs &a, uint8_t *base, int s) {
  return reinterpret_cast<float *>(base + static_cast<size_t>(a.stages) * a.piece_bytes +
                                   static_cast<size_t>(a.stages) * (a.piece_bytes / 2)) +
         static_cast<size_t>(s) * (a.piece_bytes / 256);
}

__global__ void __launch_bounds__(32) dispatch_kernel(DispatchArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ uint64_t full[kMaxStages];
  __shared__ int32_t dst[kMaxTopk];
  __shared__ int aborted;

  const int lane = threadIdx.x;
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t n_mine = first < a.nunits ? (a.nunits - 1 - first) / stride + 1 : 0;
  const int S = a.stages;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    aborted = 0;
  }
  __syncwarp();
  // The rows are inputs that layout does not write: start loading them while
  // the layout kernel may still run (programmatic dependent launch), then wait
  // for its slot ids and flags.
  if (lane == 0)
    for (int64_t i = 0; i < n_mine && i < S; ++i)
      issue_unit_load(a, dsm + static_cast<size_t>(i) * a.piece_bytes, &full[i], first + i * stride);
  grid_dependency_wait();
  if (a.early) grid_dependents_launch();

  int64_t i = 0;
  for (; i < n_mine; ++i) {
    const int s = static_cast<int>(i % S);
    const uint32_t parity = static_cast<uint32_t>((i / S) & 1);
    const int64_t unit = first + i * stride;
    const int64_t row = unit / a.pieces;
    const int piece = static_cast<int>(unit % a.pieces);
    const uint32_t off = static_cast<uint32_t>(piece) * a.piece_bytes;
    const uint32_t bytes = min(a.piece_bytes, a.row_bytes - off);

    // destinations of this row, checked against the flags of their regions
    if (lane < a.k) {
      int32_t slot = a.tok_slot[row * a.k + lane];
      if (slot >= a.nslots) {
        latch_error(a.err, MOE_EINVAL);
        slot = -1;
      } else if (slot >= 0) {
        if (wait_flag_nonzero(flag_ptr(a.parts, slot / a.max_m)) == 0) {
          latch_error(a.err, MOE_ETIMEOUT);
          slot = -1;
        }
      }
      dst[lane] = slot;
    }
    __syncwarp();

    if (piece == 0) {
      const int src = static_cast<int>(row / a.T), t = static_cast<int>(row % a.T);
      if (lane < a.k && dst[lane] >= 0) {
        const int32_t slot = dst[lane];
        int g;
        const int64_t l = slot_local(a.parts, slot, &g);
        a.parts.recv_meta[g][l] = make_int4(src, t, (slot / a.max_m) / a.R, lane);
      }
      if (a.nsc > 0 && !a.quant) {
        const float *sc = a.x_scales + row * a.nsc;
        for (int q = lane; q < a.k * a.nsc; q += 32) {
          const int j = q / a.nsc, c = q - j * a.nsc;
          const int32_t slot = dst[j];
          if (slot >= 0) {
            int g;
            const int64_t l = slot_local(a.parts, slot, &g);
            a.parts.recv_scales[g][l * a.nsc + c] = __ldg(sc + c);
          }
        }
      }
    }

    if (a.quant) {
      // every lane reads the staged bf16 piece: wait for it
      uint8_t *stage = dsm + static_cast<size_t>(s) * a.piece_bytes;
      if (!mbar_wait_bounded(&full[s], parity)) {
        latch_error(a.err, MOE_ETIMEOUT);
        aborted = 1;
      }
      __syncwarp();
      if (aborted) break;
      // the e4m3 stage of unit i - S may still be read by its bulk stores
      if (lane == 0 && i >= S) bulk_wait_read<0>();
      __syncwarp();
      uint8_t *q = qstage(a, dsm, s);
      float *qs = qscales(a, dsm, s);
      const int nblk = static_cast<int>(bytes / 256);
      quantize_blocks(reinterpret_cast<const uint16_t *>(stage), q, qs, nblk, 0, 1, lane);
      fence_proxy_async_smem();  // the shared writes above, before the bulk stores and the refill
      __syncwarp();
      const int sc0 = static_cast<int>(off / 256);
      for (int qq = lane; qq < a.k * nblk; qq += 32) {
        const int j = qq / nblk, b = qq - j * nblk;
        const int32_t slot = dst[j];
        if (slot >= 0) {
          int g;
          const int64_t l = slot_local(a.parts, slot, &g);
          a.parts.recv_scales[g][l * a.nsc + sc0 + b] = qs[b];
        }
      }
      if (lane == 0) {
        for (int j = 0; j < a.k; ++j) {
          const int32_t slot = dst[j];
          if (slot >= 0) {
            int g;
            const int64_t l = slot_local(a.parts, slot, &g);
            bulk_store(a.parts.recv_x[g] + l * (a.row_bytes / 2) + off / 2, q, bytes / 2);
          }
        }
        bulk_commit();
        // the bf16 stage has been consumed: refill it with unit i + S
        if (i + S < n_mine) issue_unit_load(a, stage, &full[s], first + (i + S) * stride);
      }
      __syncwarp();
      continue;
    }

    if (lane == 0) {
      uint8_t *stage = dsm + static_cast<size_t>(s) * a.piece_bytes;
      if (!mbar_wait_bounded(&full[s], parity)) {
        latch_error(a.err, MOE_ETIMEOUT);
        aborted = 1;
      } else {
        for (int j = 0; j < a.k; ++j) {
          const int32_t slot = dst[j];
          if (slot >= 0) {
            int g;
            const int64_t l = slot_local(a.parts, slot, &g);
            bulk_store(a.parts.recv_x[g] + l * a.row_bytes + off, stage, bytes);
          }
        }
        bulk_commit();
        // refill the stage of the previous unit once its stores have read it
        const int64_t next = i - 1 + S;
        if (i >= 1 && next < n_mine) {
          bulk_wait_read<1>();
          const int ps = static_cast<int>((i - 1) % S);
          issue_unit_load(a, dsm + static_cast<size_t>(ps) * a.piece_bytes, &full[ps], first + next * stride);
        }
      }
    }
    __syncwarp();
    if (aborted) break;
  }

  if (lane == 0) {
    if (aborted) {
      // drain the loads still in flight (bounded) before the CTA releases its shared memory
      const int64_t issued = a.quant ? (n_mine < i + S ? n_mine : i + S) : inflight_end(i, S, n_mine);
      for (int64_t u = i; u < issued; ++u)
        mbar_wait_bounded(&full[u % S], static_cast<uint32_t>((u / S) & 1));
    }
    bulk_wait_all();
  }
  __syncwarp();
}

moe_status launch_dispatch(const Sizes &s, const void *x, const float *x_scales, const int32_t *tok_slot,
                           const SlotParts &parts, int32_t *err, int num_sms, cudaStream_t stream) {
  DispatchArgs a{};
  a.x = static_cast<const uint8_t *>(x);
  a.x_scales = x_scales;
  a.tok_slot = tok_slot;
  a.parts = parts;
  a.err = err;
  a.R = s.R;
  a.T = s.T;
  a.k = s.k;
  a.max_m = s.max_m;
  a.nsc = s.nsc;
  a.early = early_trigger(s.ntok);
  a.quant = s.quant ? 1 : 0;
  a.row_bytes = static_cast<uint32_t>(s.in_row_bytes);
  a.piece_bytes = a.row_bytes < kPieceMax ? a.row_bytes : kPieceMax;  // a multiple of 256 in quant mode
  a.pieces = static_cast<int>((a.row_bytes + a.piece_bytes - 1) / a.piece_bytes);
  a.nslots = s.nslots;
  a.nunits = s.ntok * a.pieces;
  int stages = static_cast<int>(kStageBudget / a.piece_bytes);
  a.stages = stages < 2 ? 2 : (stages > kMaxStages ? kMaxStages : stages);
  if (a.nunits == 0) return MOE_OK;

  size_t smem = static_cast<size_t>(a.stages) * a.piece_bytes;
  if (a.quant) smem += static_cast<size_t>(a.stages) * (a.piece_bytes / 2 + a.piece_bytes / 256 * sizeof(float));
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return MOE_ECUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_kernel, 32, smem) != cudaSuccess)
    return MOE_ECUDA;
  if (per_sm < 1) per_sm = 1;
  const int sms = num_sms > 0 && num_sms < sm_count() ? num_sms : sm_count();
  int64_t grid = static_cast<int64_t>(sms) * per_sm;
  if (grid > a.nunits) grid = a.nunits;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  use_pdl(cfg, attr);
  if (cudaLaunchKernelEx(&cfg, dispatch_kernel, a) != cudaSuccess) return MOE_ECUDA;
  return launch_status();
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch(const moe_desc *desc, const void *x, const float *x_scales,
                                   const int32_t *tok_slot, const uint64_t *flags, void *recv_x,
                                   float *recv_scales, int32_t *recv_meta, int32_t *err, void *stream) {
  Sizes s;
  moe_status st = check_desc(desc, &s);
  if (st != MOE_OK) return st;
  if (flags == nullptr || err == nullptr || recv_x == nullptr || recv_meta == nullptr) return MOE_EINVAL;
  if (s.ntok > 0 && (x == nullptr || tok_slot == nullptr)) return MOE_EINVAL;
  if (s.dtype == MOE_FP8_E4M3) {
    if (recv_scales == nullptr || (s.ntok > 0 && x_scales == nullptr)) return MOE_EINVAL;
    if (!aligned4(x_scales) || !aligned4(recv_scales)) return MOE_EINVAL;
  } else if (s.dtype == MOE_BF16_TO_FP8) {
    if (recv_scales == nullptr || x_scales != nullptr || !aligned4(recv_scales)) return MOE_EINVAL;
  }
  if (!aligned16(x) || !aligned16(recv_x) || !aligned16(recv_meta) || !aligned4(tok_slot) || !aligned4(err))
    return MOE_EINVAL;
  return launch_dispatch(s, x, x_scales, tok_slot,
                         single_part(s, recv_x, recv_scales, recv_meta, const_cast<uint64_t *>(flags), nullptr), err,
                         desc->num_sms, static_cast<cudaStream_t>(stream));
}

/*
 * CPU oracle for MoE expert-parallel token dispatch and combine.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. This is the slow, plain,
 * single-threaded definition of what the GPU library computes. Only the tests,
 * the smoke check and the benchmark's CPU-baseline / reference arm may load it;
 * the library never does. It shares no code, header, table or helper with the
 * CUDA path: every routine below is written out from the pages' description.
 *
 * Sources (cited by title and section):
 *   [HGT]  "How GPUs Talk to Each Other During LLM Inference", section 7
 *          "Expert Parallelism".
 *   [PPLX] Perplexity, "Efficient and portable mixture-of-experts communication"
 *          (zh-TW text), sections "Introduction" (簡介), "Portable kernels"
 *          (可攜式核心), "Dispatch" (分派) and "Combine" (組合).
 *   [NVDE] "NVSHMEM and DeepEP: GPU-initiated communication", sections
 *          "High-throughput mode" (FP8 dispatch / BF16 combine bullet),
 *          "Low-latency mode: fixed slots, no CPU sync" (receive-buffer
 *          estimate) and Exercise 2 "How big should the slots be?".
 *
 * Notation: R logical EP ranks, T tokens per rank, H hidden size, E experts,
 * L = E / R local experts per rank, k experts per token, max_m slots per
 * (expert, source rank). Expert e lives on rank e / L as its local expert
 * e % L ([NVDE] high-throughput section: gpu = expert // experts-per-GPU).
 * The fixed-slot receive buffer of every rank holds, per local expert and per
 * source rank, max_m slots ([NVDE] low-latency section; [PPLX] portable
 * kernels: every sender owns a private region per expert). Concatenating the
 * ranks gives one buffer indexed by region r = e * R + src, slot
 * s = r * max_m + pos.
 *
 * Floating point: fp64 throughout; the only rounding the pages fix is that
 * combine returns BF16 ([NVDE] high-throughput section), done once at the end.
 * The expert stage ([HGT] section 7, Mega MoE: linear 1, SwiGLU, linear 2)
 * rounds its intermediate h and its output y to bf16 once each, the precision
 * the rows are stored in between the steps.
 *
 * parity pins: see the tests (brute force, invariants, closed forms, the
 * pages' printed buffer sizes, and library conversions).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
  ORC_OK = 0,
  ORC_EINVAL = -1,
  ORC_EOVERFLOW = -2,
};

/* Dispatched row formats. ORC_BF16_TO_FP8: the caller's rows are bf16 and
 * dispatch quantises them to E4M3 with 128-element fp32 scales on the way. */
enum { ORC_BF16 = 0, ORC_FP8_E4M3 = 1, ORC_BF16_TO_FP8 = 2 };

/* ------------------------------------------------------------------------ */
/* Number formats, from their definitions.                                   */
/* ------------------------------------------------------------------------ */

/* Value of a bfloat16 bit pattern: the upper half of an IEEE binary32. */
double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bfloat16 (ties to even) and return its bits.
 * bfloat16 has 8 significant bits and binary32's exponent range; in the binade
 * [2^e, 2^(e+1)) its values are spaced 2^(e-7), and below 2^-126 the spacing
 * stays 2^-133 (subnormals). rint() rounds half to even in the default mode. */
uint16_t orc_bf16_from_double(double v) {
  if (v != v) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e = ilogb(a);
  if (e < -126) e = -126;
  double quantum = scalbn(1.0, e - 7);
  double r = rint(a / quantum) * quantum;
  if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80);
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (u >> 16));
}

/* Value of an FP8 E4M3 ("e4m3fn") code: 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 is subnormal (M/8 * 2^-6); S.1111.111 is
 * NaN and there is no infinity, so the largest finite value is 448. */
double orc_e4m3_value(uint8_t code) {
  int s = code >> 7;
  int ex = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (ex == 15 && m == 7) return NAN;
  if (ex == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), ex - 10);
  return s ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Problem description and its validity.                                     */
/* ------------------------------------------------------------------------ */

/* The sizes are the pages' problem statement: tokens, routing (k of E
 * experts), logical EP ranks and the per-rank token bound max_m
 * ([PPLX] portable kernels; [NVDE] low-latency section). */
int orc_validate(int R, int T, int H, int E, int k, int max_m, int dtype) {
  if (R < 1 || T < 0 || H < 1 || E < 1 || k < 1 || max_m < 1) return ORC_EINVAL;
  if (E % R != 0) return ORC_EINVAL;       /* num_experts // EP must be exact */
  if (k > E) return ORC_EINVAL;
  if (T > max_m) return ORC_EINVAL;        /* max_m bounds tokens per rank */
  if (dtype == ORC_FP8_E4M3 || dtype == ORC_BF16_TO_FP8) {
    if (H % 128 != 0) return ORC_EINVAL;   /* one scale per 128 elements */
  } else if (dtype == ORC_BF16) {
    if (H % 8 != 0) return ORC_EINVAL;     /* rows of whole 16-byte vectors */
  } else {
    return ORC_EINVAL;
  }
  if ((int64_t)E * R * max_m > INT32_MAX) return ORC_EINVAL; /* int32 slot ids */
  if ((int64_t)R * T * k > INT32_MAX) return ORC_EINVAL;
  return ORC_OK;
}

/* Bytes of a dispatched row (in the slots) and of a caller's input row. */
static int64_t orc_row_bytes(int H, int dtype) {
  return dtype == ORC_BF16 ? (int64_t)2 * H : (int64_t)H;
}

static int64_t orc_in_row_bytes(int H, int dtype) {
  return dtype == ORC_FP8_E4M3 ? (int64_t)H : (int64_t)2 * H;
}

static int64_t orc_scale_count(int H, int dtype) {
  return dtype == ORC_BF16 ? 0 : (int64_t)H / 128;
}

/* Nearest FP8 E4M3 ("e4m3fn") code to a float, ties to even; magnitudes
 * beyond the largest finite value (448) saturate to +-448, since the format
 * has no infinity; NaN stays NaN. The representable magnitudes are m * 2^-9
 * (m = 0..7, subnormal) and (8 + m) * 2^(E - 10) for E = 1..15, except
 * E = 15, m = 7 (NaN); in the binade [2^e, 2^(e+1)) they are spaced 2^(e-3),
 * and below 2^-6 the spacing stays 2^-9. */
uint8_t orc_e4m3_from_float(float f) {
  if (f != f) return 0x7F;
  uint8_t sign = signbit(f) ? 0x80 : 0;
  double a = fabs((double)f);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a == 0.0) return sign;
  int e = ilogb(a);
  if (e < -6) e = -6;
  double quantum = scalbn(1.0, e - 3);
  double r = rint(a / quantum) * quantum;
  if (r < 0x1p-6) return (uint8_t)(sign | (uint8_t)(r / 0x1p-9)); /* subnormal */
  int E = ilogb(r);
  int m = (int)(r / scalbn(1.0, E - 3)) - 8;
  return (uint8_t)(sign | ((E + 7) << 3) | m);
}

/* Block quantisation of one bf16 row to E4M3 with one fp32 scale per 128
 * contiguous elements ("NVSHMEM and DeepEP", high-throughput section: FP8
 * dispatch with fine-grained 128-element scales). The decision of each code
 * is taken in fp32, as a GPU does it: scale = amax / 448 (1 for an all-zero
 * block), code = e4m3(x / scale) with IEEE fp32 division. */
void orc_quantize_row(const uint16_t *x, int H, uint8_t *q, float *scales) {
  for (int b = 0; b < H / 128; ++b) {
    float amax = 0.0f;
    for (int h = b * 128; h < (b + 1) * 128; ++h) {
      float v = fabsf((float)orc_bf16_value(x[h]));
      if (v > amax) amax = v;
    }
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    scales[b] = s;
    for (int h = b * 128; h < (b + 1) * 128; ++h) {
      float v = (float)orc_bf16_value(x[h]);
      q[h] = orc_e4m3_from_float(v / s);
    }
  }
}

/* Bytes of every buffer of the path for the whole allocation (all R logical
 * ranks). Per slot a receiver stores the row, its fp32 block scales and a
 * 16-byte back-index header, the message of the [NVDE] low-latency estimate
 * (hidden + hidden/128*4 + 16). Region count E*R = L*R per rank times R ranks.
 * out[0..6] = recv_x, recv_scales, recv_meta, counts, flags, tok_slot,
 * expert_out. */
int orc_buffer_sizes(int R, int T, int H, int E, int k, int max_m, int dtype,
                     int64_t *out) {
  int st = orc_validate(R, T, H, E, k, max_m, dtype);
  if (st != ORC_OK) return st;
  int64_t slots = (int64_t)E * R * max_m;
  out[0] = slots * orc_row_bytes(H, dtype);
  out[1] = slots * orc_scale_count(H, dtype) * 4;
  out[2] = slots * 16;
  out[3] = (int64_t)E * R * 4;
  out[4] = (int64_t)E * R * 8;
  out[5] = (int64_t)R * T * k * 4;
  out[6] = slots * (int64_t)H * 2;
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Layout: per-expert counts, slot of every (source rank, token, choice),    */
/* count-plus-one flags.                                                     */
/* ------------------------------------------------------------------------ */

/* [PPLX] dispatch: the sender counts, per destination expert, the tokens this
 * rank sends it and signals count + 1 (the 0 -> non-zero change means "count
 * arrived"). [NVDE] low-latency section / [PPLX] portable kernels: each sender
 * has max_m private slots per (local expert, source rank), so it can place a
 * token without talking to the receiver. Tokens are visited in order, so a
 * region's slots hold its tokens in increasing token order.
 *   topk_idx [R][T][k], counts [E][R], flags [E][R], tok_slot [R][T][k]. */
int orc_layout(int R, int T, int E, int k, int max_m, const int32_t *topk_idx,
               int32_t *counts, uint64_t *flags, int32_t *tok_slot) {
  for (int64_t r = 0; r < (int64_t)E * R; ++r) counts[r] = 0;
  for (int src = 0; src < R; ++src) {
    for (int t = 0; t < T; ++t) {
      const int32_t *row = topk_idx + ((int64_t)src * T + t) * k;
      for (int j = 0; j < k; ++j) {
        int e = row[j];
        if (e == -1) { /* a masked choice names no expert: no slot, nothing counted */
          tok_slot[((int64_t)src * T + t) * k + j] = -1;
          continue;
        }
        if (e < 0 || e >= E) return ORC_EINVAL;
        for (int jj = 0; jj < j; ++jj)
          if (row[jj] == e) return ORC_EINVAL; /* a token picks distinct experts */
        int64_t region = (int64_t)e * R + src;
        int pos = counts[region]++;
        if (pos >= max_m) return ORC_EOVERFLOW; /* slots too small: error out */
        tok_slot[((int64_t)src * T + t) * k + j] = (int32_t)(region * max_m + pos);
      }
    }
  }
  for (int64_t r = 0; r < (int64_t)E * R; ++r) flags[r] = (uint64_t)counts[r] + 1;
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Dispatch: copy each selected token into its k slots.                      */
/* ------------------------------------------------------------------------ */

/* [PPLX] dispatch: the activations, their block scales and the token's index on
 * its own rank are packed together and sent to every expert the token was
 * routed to; the receiver keeps (source rank, expert, token) for combine.
 * [NVDE]: FP8 rows carry one fp32 scale per 128 elements.
 * The fixed-slot buffer is represented sparsely: for the n_sel selected tokens
 * (flat ids src*T+t), entry i*k+j describes the slot of choice j of token
 * sel[i]: its id, its row bytes, its scales and its header
 * {source rank, token index, expert, choice j}. */
int orc_dispatch(int R, int T, int H, int E, int k, int max_m, int dtype,
                 const uint8_t *x, const float *x_scales, const int32_t *tok_slot,
                 int64_t n_sel, const int64_t *sel, int64_t *slot_id,
                 uint8_t *rows, float *scales, int32_t *meta) {
  int64_t row_bytes = orc_row_bytes(H, dtype);
  int64_t in_row_bytes = orc_in_row_bytes(H, dtype);
  int64_t nsc = orc_scale_count(H, dtype);
  int64_t nslots = (int64_t)E * R * max_m;
  uint8_t *qrow = (uint8_t *)malloc((size_t)(row_bytes > 0 ? row_bytes : 1));
  float *qsc = (float *)malloc(sizeof(float) * (size_t)(nsc > 0 ? nsc : 1));
  if (!qrow || !qsc) {
    free(qrow);
    free(qsc);
    return ORC_EINVAL;
  }
  int st = ORC_OK;
  for (int64_t i = 0; i < n_sel && st == ORC_OK; ++i) {
    int64_t tok = sel[i];
    if (tok < 0 || tok >= (int64_t)R * T) {
      st = ORC_EINVAL;
      break;
    }
    int src = (int)(tok / T), t = (int)(tok % T);
    /* the row and scales that go out: as given, or quantised once per token */
    const uint8_t *row = x + tok * in_row_bytes;
    const float *rsc = nsc > 0 && dtype == ORC_FP8_E4M3 ? x_scales + tok * nsc : qsc;
    if (dtype == ORC_BF16_TO_FP8) {
      orc_quantize_row((const uint16_t *)row, H, qrow, qsc);
      row = qrow;
    }
    for (int j = 0; j < k; ++j) {
      int64_t s = tok_slot[tok * k + j];
      if (s == -1) { /* a masked choice: nothing is sent */
        slot_id[i * k + j] = -1;
        continue;
      }
      if (s < 0 || s >= nslots) {
        st = ORC_EINVAL;
        break;
      }
      int64_t region = s / max_m;
      int e = (int)(region / R);
      if (region % R != src) { /* a slot belongs to its sender */
        st = ORC_EINVAL;
        break;
      }
      int64_t out = i * k + j;
      slot_id[out] = s;
      memcpy(rows + out * row_bytes, row, (size_t)row_bytes);
      for (int64_t b = 0; b < nsc; ++b) scales[out * nsc + b] = rsc[b];
      meta[out * 4 + 0] = src;
      meta[out * 4 + 1] = t;
      meta[out * 4 + 2] = e;
      meta[out * 4 + 3] = j;
    }
  }
  free(qrow);
  free(qsc);
  return st;
}

/* ------------------------------------------------------------------------ */
/* Receive side: compaction into contiguous expert-major buffers.            */
/* ------------------------------------------------------------------------ */

/* [PPLX] Dispatch: once the counts and payloads have arrived, the receiver
 * copies the tokens into contiguous buffers, one run per expert, which become
 * the inputs of the grouped GEMM, and keeps (source rank, expert, token) for
 * combine. Here the filled slots are packed in (expert, source rank, position)
 * order: region_offsets[r] = filled slots of the regions before r
 * (r = e * R + src), region_offsets[E * R] = total; slot s lands at packed row
 * region_offsets[s / max_m] + s % max_m. */
int orc_region_offsets(int R, int E, int max_m, const int32_t *counts, int32_t *region_offsets) {
  int64_t acc = 0;
  for (int64_t r = 0; r < (int64_t)E * R; ++r) {
    if (counts[r] < 0 || counts[r] > max_m) return ORC_EINVAL;
    region_offsets[r] = (int32_t)acc;
    acc += counts[r];
  }
  region_offsets[(int64_t)E * R] = (int32_t)acc;
  return ORC_OK;
}

/* Packed rows of n sparse slots (as produced by orc_dispatch). */
int orc_compact(int R, int E, int max_m, int64_t row_bytes, int nsc, const int32_t *region_offsets, int64_t n,
                const int64_t *slot_id, const uint8_t *rows, const float *scales, const int32_t *meta,
                int64_t n_packed, uint8_t *packed_rows, float *packed_scales, int32_t *packed_meta) {
  for (int64_t i = 0; i < n; ++i) {
    int64_t region = slot_id[i] / max_m;
    if (region < 0 || region >= (int64_t)E * R) return ORC_EINVAL;
    int64_t p = (int64_t)region_offsets[region] + slot_id[i] % max_m;
    if (p < 0 || p >= n_packed || p >= region_offsets[region + 1]) return ORC_EINVAL;
    memcpy(packed_rows + p * row_bytes, rows + i * row_bytes, (size_t)row_bytes);
    for (int b = 0; b < nsc; ++b) packed_scales[p * nsc + b] = scales[i * nsc + b];
    for (int q = 0; q < 4; ++q) packed_meta[p * 4 + q] = meta[i * 4 + q];
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* The expert stage (an expert MLP with SwiGLU) on packed rows.              */
/* ------------------------------------------------------------------------ */

/* "How GPUs Talk to Each Other During LLM Inference", section 7 (Mega MoE):
 * between dispatch and combine every expert runs linear 1, SwiGLU and linear 2
 * on its tokens. For one bf16 row x of expert e, with weights of that expert in
 * bf16 (w_gate, w_up [I][H], w_down [H][I], each row the K dimension):
 *   h[i] = bf16( silu(sum_h x[h] w_gate[i][h]) * sum_h x[h] w_up[i][h] ),
 *   silu(g) = g / (1 + exp(-g)),
 *   y[j] = bf16( sum_i h[i] w_down[j][i] ),
 * sums and silu in fp64, h rounded to bf16 once (as it is stored between the two
 * linears), y rounded once. */
/* One row through one bf16 linear map: y[n] = bf16( sum_k x[k] w[n][k] ) for a
 * weight matrix w [N][K] (each row one output, K contiguous), fp64 sum. This is
 * linear 2 of the expert stage on its own. */
void orc_linear_row(int K, int N, const uint16_t *x, const uint16_t *w, uint16_t *y) {
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int k = 0; k < K; ++k) acc += orc_bf16_value(x[k]) * orc_bf16_value(w[(int64_t)n * K + k]);
    y[n] = orc_bf16_from_double(acc);
  }
}

void orc_expert_mlp_row(int H, int I, const uint16_t *x, const uint16_t *w_gate, const uint16_t *w_up,
                        const uint16_t *w_down, uint16_t *h, uint16_t *y) {
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int k = 0; k < H; ++k) {
      double xv = orc_bf16_value(x[k]);
      g += xv * orc_bf16_value(w_gate[(int64_t)i * H + k]);
      u += xv * orc_bf16_value(w_up[(int64_t)i * H + k]);
    }
    h[i] = orc_bf16_from_double(g / (1.0 + exp(-g)) * u);
  }
  for (int j = 0; j < H; ++j) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += orc_bf16_value(h[i]) * orc_bf16_value(w_down[(int64_t)j * I + i]);
    y[j] = orc_bf16_from_double(acc);
  }
}

/* The fp8 expert stage. Rows arrive as e4m3 codes with one fp32 scale per 128
 * contiguous elements (the dispatch format, "NVSHMEM and DeepEP", high-throughput
 * section). Weights are e4m3 codes with one fp32 scale per 128 x 128 block
 * (rows n, columns k: scale ws[n / 128][k / 128]). Every value is its code
 * times its scale, and the products and sums are taken in fp64. */

/* y[n] = bf16( sum_k x[k] w[n][k] ) for one fp8 row x (K codes, K/128 scales)
 * through an fp8 weight matrix w [N][K] with block scales [N/128][K/128]. */
void orc_linear_row_fp8(int K, int N, const uint8_t *xq, const float *xs, const uint8_t *wq, const float *ws,
                        uint16_t *y) {
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int k = 0; k < K; ++k) {
      double xv = orc_e4m3_value(xq[k]) * (double)xs[k / 128];
      double wv = orc_e4m3_value(wq[(int64_t)n * K + k]) * (double)ws[(int64_t)(n / 128) * (K / 128) + k / 128];
      acc += xv * wv;
    }
    y[n] = orc_bf16_from_double(acc);
  }
}

/* Linear 1 with SwiGLU for one fp8 row, h block-quantised for linear 2:
 *   hv[i] = silu(g) * u (fp64), g and u the fp8 dot products with the gate and
 *   up rows of the expert; then per 128 contiguous i, with hv rounded to fp32
 *   (the precision the decision is taken in, as for dispatch): scale =
 *   amax / 448 (1 for an all-zero block), code = e4m3(hv / scale), fp32 IEEE
 *   division. hv (fp64) is returned too, for the callers' error bars. */
void orc_gate_up_row_fp8(int H, int I, const uint8_t *xq, const float *xs, const uint8_t *wgq, const float *wgs,
                         const uint8_t *wuq, const float *wus, double *hv, uint8_t *hq, float *hs) {
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int k = 0; k < H; ++k) {
      double xv = orc_e4m3_value(xq[k]) * (double)xs[k / 128];
      int64_t sb = (int64_t)(i / 128) * (H / 128) + k / 128;
      g += xv * orc_e4m3_value(wgq[(int64_t)i * H + k]) * (double)wgs[sb];
      u += xv * orc_e4m3_value(wuq[(int64_t)i * H + k]) * (double)wus[sb];
    }
    hv[i] = g / (1.0 + exp(-g)) * u;
  }
  for (int b = 0; b < I / 128; ++b) {
    float amax = 0.0f;
    for (int i = b * 128; i < (b + 1) * 128; ++i) {
      float v = fabsf((float)hv[i]);
      if (v > amax) amax = v;
    }
    float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    hs[b] = sc;
    for (int i = b * 128; i < (b + 1) * 128; ++i) hq[i] = orc_e4m3_from_float((float)hv[i] / sc);
  }
}

/* ------------------------------------------------------------------------ */
/* Cross-node traffic of a routing (per-node deduplication accounting).      */
/* ------------------------------------------------------------------------ */

/* [NVDE] high-throughput section: a token of a GPU on node n goes to the nodes of
 * its k experts; counting the copies that leave node n per expert, per distinct
 * destination GPU, or per distinct destination node (DeepEP's per-node
 * deduplication) gives the cross-node traffic of the three schemes. Ranks are
 * grouped ranks_per_node to a node; expert e lives on rank e / (E / R).
 * stats[src * 4 + 0..3] = tokens, per-expert, per-rank, per-node copies of
 * source rank src, summed over its tokens. */
int orc_route_stats(int R, int T, int E, int k, int ranks_per_node, const int32_t *topk_idx, int64_t *stats) {
  if (ranks_per_node < 1 || E % R != 0) return ORC_EINVAL;
  int L = E / R;
  for (int src = 0; src < R; ++src) {
    int64_t per_expert = 0, per_rank = 0, per_node = 0;
    int home = src / ranks_per_node;
    for (int t = 0; t < T; ++t) {
      const int32_t *row = topk_idx + ((int64_t)src * T + t) * k;
      for (int j = 0; j < k; ++j) {
        if (row[j] == -1) continue; /* a masked choice sends nothing */
        if (row[j] < 0 || row[j] >= E) return ORC_EINVAL;
        int rank = row[j] / L, node = rank / ranks_per_node;
        if (node == home) continue;
        per_expert += 1;
        int seen_rank = 0, seen_node = 0; /* first choice with this rank / node? */
        for (int jj = 0; jj < j; ++jj) {
          if (row[jj] == -1) continue;
          int r2 = row[jj] / L;
          if (r2 == rank) seen_rank = 1;
          if (r2 / ranks_per_node == node) seen_node = 1;
        }
        per_rank += !seen_rank;
        per_node += !seen_node;
      }
    }
    stats[src * 4 + 0] = T;
    stats[src * 4 + 1] = per_expert;
    stats[src * 4 + 2] = per_rank;
    stats[src * 4 + 3] = per_node;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Synthetic experts (not part of the pages' method: a stand-in for the      */
/* expert MLPs that run between dispatch and combine).                       */
/* ------------------------------------------------------------------------ */

/* FP8 rows: y = bf16( q * scale * (1 + e/256) ) per element, with q the E4M3
 * value, scale its 128-element block scale and e the slot's expert. The product
 * is exact in fp64 (4 x 24 x 9 significant bits), so it is rounded once.
 * BF16 rows: identity (y = the row). */
int orc_expert_stub(int R, int H, int E, int max_m, int dtype, int64_t n,
                    const int64_t *slot_id, const uint8_t *rows, const float *scales,
                    uint16_t *y) {
  int64_t row_bytes = orc_row_bytes(H, dtype);
  int64_t nsc = orc_scale_count(H, dtype);
  for (int64_t i = 0; i < n; ++i) {
    int64_t region = slot_id[i] / max_m;
    int e = (int)(region / R);
    if (e < 0 || e >= E) return ORC_EINVAL;
    const uint8_t *row = rows + i * row_bytes;
    uint16_t *yo = y + i * (int64_t)H;
    if (dtype != ORC_BF16) {
      double c = 1.0 + (double)e / 256.0;
      for (int h = 0; h < H; ++h) {
        double v = orc_e4m3_value(row[h]) * (double)scales[i * nsc + h / 128] * c;
        yo[h] = orc_bf16_from_double(v);
      }
    } else {
      memcpy(yo, row, (size_t)H * 2);
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Combine: weighted sum of each token's k expert outputs, back in the       */
/* token's own order.                                                        */
/* ------------------------------------------------------------------------ */

typedef struct {
  int64_t slot;
  int64_t index;
} orc_slot_ref;

static int orc_cmp_slot(const void *a, const void *b) {
  int64_t x = ((const orc_slot_ref *)a)->slot, y = ((const orc_slot_ref *)b)->slot;
  return (x > y) - (x < y);
}

/* [HGT] section 7 and [PPLX] introduction: the layer output of a token is the
 * sum over its k experts of expert output times the router weight of that
 * expert. [PPLX] combine: the receiver finds, through the routing table, which
 * slot to read for each expert and which weight to apply, and writes the
 * weighted sum into a caller-allocated tensor. The weights are applied at the
 * receiver, in fp64, and the sum is rounded to bf16 once. The sum starts from
 * its first term (not from a +0 accumulator), so a token whose terms are all
 * -0 keeps the sign of its zeros, as a sum of those terms does.
 *   y: n_slots rows of H bf16, row i being the expert output of slot slot_id[i];
 *   out: n_sel rows of H bf16 for the selected tokens sel[]. */
int orc_combine(int R, int T, int H, int E, int k, int max_m, int64_t n_sel,
                const int64_t *sel, const int32_t *tok_slot, const float *weights,
                int64_t n_slots, const int64_t *slot_id, const uint16_t *y,
                uint16_t *out) {
  (void)E;
  (void)max_m;
  orc_slot_ref *index = (orc_slot_ref *)malloc(sizeof(orc_slot_ref) * (size_t)(n_slots > 0 ? n_slots : 1));
  double *acc = (double *)malloc(sizeof(double) * (size_t)H);
  if (!index || !acc) {
    free(index);
    free(acc);
    return ORC_EINVAL;
  }
  for (int64_t i = 0; i < n_slots; ++i) {
    index[i].slot = slot_id[i];
    index[i].index = i;
  }
  qsort(index, (size_t)n_slots, sizeof(orc_slot_ref), orc_cmp_slot);
  int st = ORC_OK;
  for (int64_t i = 0; i < n_sel && st == ORC_OK; ++i) {
    int64_t tok = sel[i];
    if (tok < 0 || tok >= (int64_t)R * T) {
      st = ORC_EINVAL;
      break;
    }
    for (int j = 0; j < k; ++j) {
      if (tok_slot[tok * k + j] == -1) { /* a masked choice is a zero term */
        for (int h = 0; h < H; ++h) acc[h] = (j == 0) ? 0.0 : acc[h] + 0.0;
        continue;
      }
      orc_slot_ref key = {tok_slot[tok * k + j], 0};
      const orc_slot_ref *hit = (const orc_slot_ref *)bsearch(
          &key, index, (size_t)n_slots, sizeof(orc_slot_ref), orc_cmp_slot);
      if (!hit) {
        st = ORC_EINVAL;
        break;
      }
      double w = (double)weights[tok * k + j];
      const uint16_t *yr = y + hit->index * (int64_t)H;
      for (int h = 0; h < H; ++h) {
        double term = w * orc_bf16_value(yr[h]);
        acc[h] = (j == 0) ? term : acc[h] + term; /* a sum of the k terms, no extra +0 */
      }
    }
    for (int h = 0; h < H; ++h) out[i * (int64_t)H + h] = orc_bf16_from_double(acc[h]);
  }
  free(index);
  free(acc);
  return st;
}

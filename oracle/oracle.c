/*
 * oracle.c -- plain, slow fp64 CPU reference for the fused MoE expert layer
 * with per-token multi-LoRA adapters.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file or the library built from it; only the tests, the smoke
 * check and the benchmark's CPU-baseline leg do.  It shares no code, header,
 * table or helper with the CUDA library: every step below is written out from
 * the definitions on the source pages, with no blocking, fusion or
 * reordering beyond what those definitions state.
 *
 * Sources (pages this implements):
 *  [P1] "Amazon SageMaker 및 Amazon Bedrock에서 vLLM을 활용한 MoE 모델 Multi-LoRA
 *       서빙 최적화" (aitrends.kr), section "섹션별 상세" paragraph 1 (the LoRA
 *       shrink and expand are folded into each expert's projection) and
 *       section "이미지 분석 / Diagram" (an adapter path on both the gate_up
 *       and the down projection).
 *  [P3] "[vllm] vLLM ROCm 환경에서 Shared-Expert Fusion을 통한 MoE 추론 성능
 *       최적화" (blog.secrett2633.cloud), section "코드 분석" items 1 (shared
 *       experts appended after the routed top-k slots, ids starting at the
 *       routed expert count, weight shared_expert_weight) and 2 (align runs
 *       over w13.shape[0] experts), and section "교훈" item 2 (the shared
 *       weight 1/routed_scaling_factor keeps the fused form equal to the
 *       separate shared MLP).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - activation: plain SwiGLU silu(g)*u, w13 rows [0,I) are gate, [I,2I) up;
 *  - one LoRA pair per (adapter, expert) on gate_up (A13 [r,H], B13 [2I,r])
 *    and on down (A2 [r,I], B2 [H,r]); the delta s*B(Ax) is added to the
 *    projection output before SwiGLU / before the combine;
 *  - top-k order: descending key, ties to the lower expert id;
 *  - softmax routing selects on the raw logits (monotone in the softmax) and
 *    weights by the softmax of the selected logits when renormalising, else
 *    by the full softmax;
 *  - sigmoid+bias routing selects on sigmoid(l)+b, computed in fp32 (the
 *    precision the GPU takes the same integer decision in), and weights by
 *    sigmoid(l) (bias-free), renormalised over the routed slots only;
 *  - align: experts in ascending id, slots of one expert in ascending flat
 *    slot index f = m*K' + k, each expert's list padded with the sentinel
 *    M*K' to a multiple of block_m; the tail of sorted_ids beyond the padded
 *    total is the sentinel and the tail of expert_ids is -1;
 *  - token_lora_idx outside [-1, L) is treated as -1 (no adapter).
 *
 * Bf16 tensors arrive as raw 16-bit patterns and are widened exactly to
 * double.  All arithmetic is double precision except the fp32 routing key.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Is candidate (key_a, id_a) ranked before (key_b, id_b)?  Descending key,
 * ties to the lower id. */
static int ranks_before_f(float key_a, int id_a, float key_b, int id_b) {
    if (key_a != key_b) return key_a > key_b;
    return id_a < id_b;
}

/*
 * Top-k routing with forced shared-expert slots ([P3] "코드 분석" 1).
 * Output per token: K' = top_k + n_shared ids and weights.  Routed slots
 * k < top_k hold the selected experts in rank order; shared slot top_k + j
 * holds expert E + j with weight 1/routed_scaling_factor ([P3] "교훈" 2).
 * Weights are returned in double.
 */
int oracle_moe_route(const float* logits, const float* bias, int M, int E,
                     int top_k, int scoring, int renormalize, int n_shared,
                     float routed_scaling_factor, int32_t* topk_ids,
                     double* topk_w) {
    if (M < 0 || E <= 0 || top_k <= 0 || top_k > E || n_shared < 0) return ORACLE_BAD_ARG;
    if (scoring != 0 && scoring != 1) return ORACLE_BAD_ARG;
    if (n_shared > 0 && !(routed_scaling_factor > 0.0f)) return ORACLE_BAD_ARG;
    const int KT = top_k + n_shared;
    float* key = (float*)malloc(sizeof(float) * (size_t)E);
    int* taken = (int*)malloc(sizeof(int) * (size_t)E);
    if (!key || !taken) { free(key); free(taken); return ORACLE_BAD_ARG; }
    for (int m = 0; m < M; ++m) {
        const float* l = logits + (size_t)m * E;
        for (int e = 0; e < E; ++e) {
            if (scoring == 0) {
                key[e] = l[e];
            } else {
                /* the routing decision is an integer taken in fp32 */
                float sg = 1.0f / (1.0f + expf(-l[e]));
                key[e] = sg + (bias ? bias[e] : 0.0f);
            }
            taken[e] = 0;
        }
        int32_t* ids = topk_ids + (size_t)m * KT;
        double* w = topk_w + (size_t)m * KT;
        /* selection: k passes, each taking the best remaining candidate */
        for (int k = 0; k < top_k; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before_f(key[e], e, key[best], best)) best = e;
            }
            taken[best] = 1;
            ids[k] = best;
        }
        if (scoring == 0) {
            double lmax = -INFINITY;
            for (int e = 0; e < E; ++e) if ((double)l[e] > lmax) lmax = (double)l[e];
            double denom = 0.0;
            if (renormalize) {
                for (int k = 0; k < top_k; ++k) denom += exp((double)l[ids[k]] - lmax);
            } else {
                for (int e = 0; e < E; ++e) denom += exp((double)l[e] - lmax);
            }
            for (int k = 0; k < top_k; ++k) w[k] = exp((double)l[ids[k]] - lmax) / denom;
        } else {
            double sum = 0.0;
            for (int k = 0; k < top_k; ++k) {
                w[k] = 1.0 / (1.0 + exp(-(double)l[ids[k]]));
                sum += w[k];
            }
            if (renormalize) for (int k = 0; k < top_k; ++k) w[k] /= sum;
        }
        for (int j = 0; j < n_shared; ++j) {
            ids[top_k + j] = E + j;
            w[top_k + j] = 1.0 / (double)routed_scaling_factor;
        }
    }
    free(key);
    free(taken);
    return ORACLE_OK;
}

/* Upper bound of the padded length: every non-empty expert adds at most
 * block_m - 1 sentinels, and there are at most min(E_tot, M*K') of them. */
long oracle_moe_align_max_padded(int M, int K_total, int E_tot, int block_m) {
    long slots = (long)M * K_total;
    long nonempty = slots < E_tot ? slots : E_tot;
    long bound = slots + nonempty * (block_m - 1);
    return (bound + block_m - 1) / block_m * block_m;
}

/*
 * Sort and pad slots by expert ([P3] "코드 분석" 2: over E_tot =
 * w13.shape[0] experts, shared ones included).
 */
int oracle_moe_align(const int32_t* topk_ids, int M, int K_total, int E_tot,
                     int block_m, int32_t* sorted_ids, int32_t* expert_ids,
                     int32_t* num_post_padded) {
    if (M < 0 || K_total <= 0 || E_tot <= 0 || block_m <= 0) return ORACLE_BAD_ARG;
    const long slots = (long)M * K_total;
    const long max_padded = oracle_moe_align_max_padded(M, K_total, E_tot, block_m);
    const int32_t sentinel = (int32_t)slots;
    long pos = 0;
    for (int e = 0; e < E_tot; ++e) {
        long start = pos;
        for (long f = 0; f < slots; ++f)
            if (topk_ids[f] == e) sorted_ids[pos++] = (int32_t)f;
        while ((pos - start) % block_m != 0) sorted_ids[pos++] = sentinel;
        for (long b = start / block_m; b < pos / block_m; ++b) expert_ids[b] = e;
    }
    *num_post_padded = (int32_t)pos;
    for (long p = pos; p < max_padded; ++p) sorted_ids[p] = sentinel;
    for (long b = pos / block_m; b < max_padded / block_m; ++b) expert_ids[b] = -1;
    return ORACLE_OK;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * One expert applied to one token, with the token's adapter folded into both
 * projections ([P1] "섹션별 상세" 1, "Diagram").  Writes d[0..H).
 * scratch must hold 2I + I + 2r doubles.
 */
static void expert_with_lora(const double* xm, const uint16_t* w13, const uint16_t* w2,
                             const uint16_t* A13, const uint16_t* B13,
                             const uint16_t* A2, const uint16_t* B2,
                             int e, int l, int H, int I, int E_tot, int r,
                             double scaling, double* scratch, double* d) {
    double* h = scratch;          /* [2I]: gate then up */
    double* a = h + 2 * (size_t)I; /* [I]  */
    double* t = a + I;            /* [r]  */
    double* t2 = t + r;           /* [r]  */
    const uint16_t* W13 = w13 + (size_t)e * 2 * I * H;
    for (int j = 0; j < 2 * I; ++j) {
        double s = 0.0;
        for (int i = 0; i < H; ++i) s += xm[i] * bf16_bits_to_double(W13[(size_t)j * H + i]);
        h[j] = s;
    }
    if (l >= 0) {
        const uint16_t* A = A13 + ((size_t)l * E_tot + e) * r * H;
        const uint16_t* B = B13 + ((size_t)l * E_tot + e) * 2 * I * r;
        for (int q = 0; q < r; ++q) {
            double s = 0.0;
            for (int i = 0; i < H; ++i) s += xm[i] * bf16_bits_to_double(A[(size_t)q * H + i]);
            t[q] = s;
        }
        for (int j = 0; j < 2 * I; ++j) {
            double s = 0.0;
            for (int q = 0; q < r; ++q) s += t[q] * bf16_bits_to_double(B[(size_t)j * r + q]);
            h[j] += scaling * s;
        }
    }
    for (int j = 0; j < I; ++j) a[j] = silu(h[j]) * h[I + j];
    const uint16_t* W2 = w2 + (size_t)e * H * I;
    for (int o = 0; o < H; ++o) {
        double s = 0.0;
        for (int j = 0; j < I; ++j) s += a[j] * bf16_bits_to_double(W2[(size_t)o * I + j]);
        d[o] = s;
    }
    if (l >= 0) {
        const uint16_t* A = A2 + ((size_t)l * E_tot + e) * r * I;
        const uint16_t* B = B2 + ((size_t)l * E_tot + e) * H * r;
        for (int q = 0; q < r; ++q) {
            double s = 0.0;
            for (int j = 0; j < I; ++j) s += a[j] * bf16_bits_to_double(A[(size_t)q * I + j]);
            t2[q] = s;
        }
        for (int o = 0; o < H; ++o) {
            double s = 0.0;
            for (int q = 0; q < r; ++q) s += t2[q] * bf16_bits_to_double(B[(size_t)o * r + q]);
            d[o] += scaling * s;
        }
    }
}

/*
 * The layer: y[m] = out_scale * sum_k topk_w[m,k] * Expert_{topk_ids[m,k]}(x[m])
 * with token m's adapter l = token_lora_idx[m] applied inside every expert
 * (l = -1: none).  A LoRA pointer set of NULL (or L == 0) means no adapters.
 * y is written in double, [M, H].
 */
int oracle_moe_forward(const uint16_t* x, const uint16_t* w13, const uint16_t* w2,
                       const uint16_t* A13, const uint16_t* B13,
                       const uint16_t* A2, const uint16_t* B2,
                       const int32_t* token_lora_idx, const int32_t* topk_ids,
                       const float* topk_w, int M, int H, int I, int E_tot,
                       int K_total, int L, int r, float scaling,
                       float out_scale, double* y) {
    if (M < 0 || H <= 0 || I <= 0 || E_tot <= 0 || K_total <= 0 || L < 0 || r < 0)
        return ORACLE_BAD_ARG;
    const int has_lora = A13 && B13 && A2 && B2 && token_lora_idx && L > 0 && r > 0;
    int bad = 0;
#pragma omp parallel
    {
        double* xm = (double*)malloc(sizeof(double) * (size_t)H);
        double* d = (double*)malloc(sizeof(double) * (size_t)H);
        double* acc = (double*)malloc(sizeof(double) * (size_t)H);
        double* scratch = (double*)malloc(sizeof(double) * (3 * (size_t)I + 2 * (size_t)(r > 0 ? r : 1)));
        if (!xm || !d || !acc || !scratch) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int m = 0; m < M; ++m) {
                int l = has_lora ? token_lora_idx[m] : -1;
                if (l < -1 || l >= L) l = -1;
                for (int i = 0; i < H; ++i) xm[i] = bf16_bits_to_double(x[(size_t)m * H + i]);
                for (int o = 0; o < H; ++o) acc[o] = 0.0;
                for (int k = 0; k < K_total; ++k) {
                    int e = topk_ids[(size_t)m * K_total + k];
                    double w = (double)topk_w[(size_t)m * K_total + k];
                    if (e < 0 || e >= E_tot) {
#pragma omp atomic write
                        bad = 1;
                        continue;
                    }
                    expert_with_lora(xm, w13, w2, A13, B13, A2, B2, e, l, H, I, E_tot, r,
                                     (double)scaling, scratch, d);
                    for (int o = 0; o < H; ++o) acc[o] += w * d[o];
                }
                for (int o = 0; o < H; ++o) y[(size_t)m * H + o] = (double)out_scale * acc[o];
            }
        }
        free(xm);
        free(d);
        free(acc);
        free(scratch);
    }
    return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* ------------------------------------------------------------------ MXFP8 --
 * The layer with MXFP8 expert weights.  [P3] "코드 분석" item 2 names the
 * experts implementation the fused layer runs on (an "mxfp8 native" MoE);
 * the pages do not define the format, so it is taken from the OCP
 * Microscaling (MX) Formats Specification v1.0, MXFP8 with E4M3 elements:
 *  - a block is 32 consecutive elements along the reduction dimension (H for
 *    the gate_up weights and for x, I for the down weights and for the
 *    SwiGLU output); it shares one E8M0 scale 2^(s - 127), s in [0, 254];
 *  - each element is FP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa
 *    bits, subnormals m * 2^-9, no infinity, largest finite 448;
 *  - conversion of a block (the specification's section on converting a
 *    vector to an MX format): the shared exponent is floor(log2(max |v|))
 *    minus 8 (8 = the exponent of E4M3's largest normal), clamped to the
 *    E8M0 range; each element is v / 2^shared rounded to the nearest E4M3
 *    value, ties to even, and saturated to +-448.  A block of zeros gets the
 *    smallest scale.
 * Readings (not fixed by the pages): the expert weights and the activations
 * that meet them (x for gate_up, the SwiGLU output for down) are MXFP8;
 * the LoRA adapters stay bf16 and read the unquantized activations, as in
 * the bf16 layer, and the gate_up adapter's shrink result s * (x A13^T)
 * enters its expand as a bf16 value (rounded to nearest even, through
 * fp32).  That rounding decides values which the SwiGLU output's MXFP8
 * quantization then turns into codes -- a decision that both sides must
 * take from the same numbers.  Everything else is fp64, as above.
 */
/* fp64 -> fp32 -> bf16, each step rounded to nearest even. */
static double bf16_round(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}
static double e4m3_value(uint8_t b) {
    const int s = b >> 7, E = (b >> 3) & 15, m = b & 7;
    double v;
    if (E == 15 && m == 7) return NAN;
    if (E == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, E - 7);
    return s ? -v : v;
}

/* Nearest E4M3 value to v (ties to even), saturated to +-448; the sign of
 * zero is kept. */
static uint8_t e4m3_code(double v) {
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs(v);
    if (!(a < 448.0)) return sign | 0x7E;
    int e;
    if (a < ldexp(1.0, -6)) {
        e = -6; /* subnormals share the smallest normal exponent's step */
    } else {
        frexp(a, &e);
        e -= 1; /* a in [2^e, 2^(e+1)) */
    }
    const double step = ldexp(1.0, e - 3);
    const double q = rint(a / step) * step; /* round to nearest, ties to even */
    if (q == 0.0) return sign;
    if (q < ldexp(1.0, -6)) return sign | (uint8_t)(q / ldexp(1.0, -9));
    int E;
    frexp(q, &E);
    E -= 1;
    const int m = (int)((q / ldexp(1.0, E) - 1.0) * 8.0);
    return sign | (uint8_t)(((E + 7) << 3) | m);
}

/* One block of 32 values to E4M3 codes and its E8M0 scale byte. */
static void mx_block(const double* v, uint8_t* codes, uint8_t* scale) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i)
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
    int se = -127;
    if (amax > 0.0) {
        int e;
        frexp(amax, &e);
        se = (e - 1) - 8;
        if (se < -127) se = -127;
        if (se > 127) se = 127;
    }
    *scale = (uint8_t)(se + 127);
    const double inv = ldexp(1.0, -se);
    for (int i = 0; i < 32; ++i) codes[i] = e4m3_code(v[i] * inv);
}

/* MXFP8 of a bf16 matrix [rows, K] (K a multiple of 32): codes [rows, K],
 * scales [rows, K/32]. */
int oracle_mx_quantize(const uint16_t* w, long rows, int K, uint8_t* codes, uint8_t* scales) {
    if (rows < 0 || K <= 0 || K % 32) return ORACLE_BAD_ARG;
    /* rows are independent: one per thread at a time */
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        double v[32];
        for (int b = 0; b < K / 32; ++b) {
            for (int i = 0; i < 32; ++i) v[i] = bf16_bits_to_double(w[r * K + b * 32 + i]);
            mx_block(v, codes + r * K + b * 32, scales + r * (K / 32) + b);
        }
    }
    return ORACLE_OK;
}

/* The values an MXFP8 matrix stands for: code value * 2^(scale - 127). */
int oracle_mx_dequantize(const uint8_t* codes, const uint8_t* scales, long rows, int K, double* out) {
    if (rows < 0 || K <= 0 || K % 32) return ORACLE_BAD_ARG;
    for (long r = 0; r < rows; ++r)
        for (int k = 0; k < K; ++k)
            out[r * K + k] = e4m3_value(codes[r * K + k]) * ldexp(1.0, (int)scales[r * (K / 32) + k / 32] - 127);
    return ORACLE_OK;
}

/* A vector quantized to MXFP8 and read back: n a multiple of 32. */
static void mx_round_trip(const double* v, int n, double* out) {
    uint8_t c[32], s;
    for (int b = 0; b < n / 32; ++b) {
        mx_block(v + b * 32, c, &s);
        for (int i = 0; i < 32; ++i) out[b * 32 + i] = e4m3_value(c[i]) * ldexp(1.0, (int)s - 127);
    }
}

/*
 * One expert on one token with MXFP8 weights ([P1] "섹션별 상세" 1,
 * "Diagram": the adapter on both projections; the adapter reads the
 * unquantized activations).  xq: the token's x through MXFP8, xm: x itself.
 * wv: a 256-entry table of E4M3 code values, sv: of E8M0 scales.
 */
static void expert_mx(const double* xq, const double* xm, const uint8_t* w13q, const uint8_t* w13s,
                      const uint8_t* w2q, const uint8_t* w2s, const uint16_t* A13, const uint16_t* B13,
                      const uint16_t* A2, const uint16_t* B2, int e, int l, int H, int I, int E_tot, int r,
                      double scaling, const double* wv, const double* sv, double* scratch, double* dout) {
    double* hh = scratch;             /* [2I] gate then up */
    double* act = hh + 2 * (size_t)I; /* [I] SwiGLU output */
    double* actq = act + I;           /* [I] the same through MXFP8 */
    double* ts = actq + I;            /* [r] gate_up shrink */
    double* ts2 = ts + r;             /* [r] down shrink */
    const uint8_t* Q13 = w13q + (size_t)e * 2 * I * H;
    const uint8_t* S13 = w13s + (size_t)e * 2 * I * (H / 32);
    for (int j = 0; j < 2 * I; ++j) {
        double acc_j = 0.0;
        for (int i = 0; i < H; ++i)
            acc_j += xq[i] * wv[Q13[(size_t)j * H + i]] * sv[S13[(size_t)j * (H / 32) + i / 32]];
        hh[j] = acc_j;
    }
    if (l >= 0) {
        const uint16_t* Ash = A13 + ((size_t)l * E_tot + e) * r * H;
        const uint16_t* Bex = B13 + ((size_t)l * E_tot + e) * 2 * I * r;
        for (int q = 0; q < r; ++q) {
            double acc_q = 0.0;
            for (int i = 0; i < H; ++i) acc_q += xm[i] * bf16_bits_to_double(Ash[(size_t)q * H + i]);
            ts[q] = bf16_round(scaling * acc_q);
        }
        for (int j = 0; j < 2 * I; ++j) {
            double acc_j = 0.0;
            for (int q = 0; q < r; ++q) acc_j += ts[q] * bf16_bits_to_double(Bex[(size_t)j * r + q]);
            hh[j] += acc_j;
        }
    }
    for (int j = 0; j < I; ++j) act[j] = silu(hh[j]) * hh[I + j];
    mx_round_trip(act, I, actq);
    const uint8_t* Q2 = w2q + (size_t)e * H * I;
    const uint8_t* S2 = w2s + (size_t)e * H * (I / 32);
    for (int o = 0; o < H; ++o) {
        double acc_o = 0.0;
        for (int j = 0; j < I; ++j)
            acc_o += actq[j] * wv[Q2[(size_t)o * I + j]] * sv[S2[(size_t)o * (I / 32) + j / 32]];
        dout[o] = acc_o;
    }
    if (l >= 0) {
        const uint16_t* Ash = A2 + ((size_t)l * E_tot + e) * r * I;
        const uint16_t* Bex = B2 + ((size_t)l * E_tot + e) * H * r;
        for (int q = 0; q < r; ++q) {
            double acc_q = 0.0;
            for (int j = 0; j < I; ++j) acc_q += act[j] * bf16_bits_to_double(Ash[(size_t)q * I + j]);
            ts2[q] = acc_q;
        }
        for (int o = 0; o < H; ++o) {
            double acc_o = 0.0;
            for (int q = 0; q < r; ++q) acc_o += ts2[q] * bf16_bits_to_double(Bex[(size_t)o * r + q]);
            dout[o] += scaling * acc_o;
        }
    }
}

/*
 * The layer with MXFP8 expert weights: as oracle_moe_forward, with w13 given
 * as codes [E_tot, 2I, H] and scales [E_tot, 2I, H/32], w2 as codes
 * [E_tot, H, I] and scales [E_tot, H, I/32]; H and I multiples of 32.
 */
int oracle_moe_forward_mx(const uint16_t* x, const uint8_t* w13q, const uint8_t* w13s, const uint8_t* w2q,
                          const uint8_t* w2s, const uint16_t* A13, const uint16_t* B13, const uint16_t* A2,
                          const uint16_t* B2, const int32_t* token_lora_idx, const int32_t* topk_ids,
                          const float* topk_w, int M, int H, int I, int E_tot, int K_total, int L, int r,
                          float scaling, float out_scale, double* y) {
    if (M < 0 || H <= 0 || I <= 0 || H % 32 || I % 32 || E_tot <= 0 || K_total <= 0 || L < 0 || r < 0)
        return ORACLE_BAD_ARG;
    const int has_lora = A13 && B13 && A2 && B2 && token_lora_idx && L > 0 && r > 0;
    double wv[256], sv[256];
    for (int b = 0; b < 256; ++b) {
        wv[b] = e4m3_value((uint8_t)b);
        sv[b] = ldexp(1.0, b - 127);
    }
    int bad = 0;
#pragma omp parallel
    {
        double* xm = (double*)malloc(sizeof(double) * (size_t)H);
        double* xq = (double*)malloc(sizeof(double) * (size_t)H);
        double* d = (double*)malloc(sizeof(double) * (size_t)H);
        double* acc = (double*)malloc(sizeof(double) * (size_t)H);
        double* scratch = (double*)malloc(sizeof(double) * (4 * (size_t)I + 2 * (size_t)(r > 0 ? r : 1)));
        if (!xm || !xq || !d || !acc || !scratch) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int m = 0; m < M; ++m) {
                int l = has_lora ? token_lora_idx[m] : -1;
                if (l < -1 || l >= L) l = -1;
                for (int i = 0; i < H; ++i) xm[i] = bf16_bits_to_double(x[(size_t)m * H + i]);
                mx_round_trip(xm, H, xq);
                for (int o = 0; o < H; ++o) acc[o] = 0.0;
                for (int k = 0; k < K_total; ++k) {
                    int e = topk_ids[(size_t)m * K_total + k];
                    double w = (double)topk_w[(size_t)m * K_total + k];
                    if (e < 0 || e >= E_tot) {
#pragma omp atomic write
                        bad = 1;
                        continue;
                    }
                    expert_mx(xq, xm, w13q, w13s, w2q, w2s, A13, B13, A2, B2, e, l, H, I, E_tot, r,
                              (double)scaling, wv, sv, scratch, d);
                    for (int o = 0; o < H; ++o) acc[o] += d[o] * w;
                }
                for (int o = 0; o < H; ++o) y[(size_t)m * H + o] = acc[o] * (double)out_scale;
            }
        }
        free(xm);
        free(xq);
        free(d);
        free(acc);
        free(scratch);
    }
    return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

// MoE-layer oracle (forward and backward): plain, slow, fp64 CPU code.
//
// TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
// CPU-baseline leg load this library. The product path (the CUDA library under
// mixture_experts_layer_gemv_gb300/csrc) shares no code, header, table or helper
// with it, and neither side includes or links the other.
//
// What it computes, step by step, follows the DeepSeek-V2 MoE stages as described
// on "DSV2-236B-MegaKernel" (README, stage flowchart, MoE subgraph, stages M..R):
//   M  RMSNorm in front of the router (optional: the fused-norm entry points)
//   N  router GEMV            logits = W_router . x                      (fp64 here)
//   O  softmax + group-limited greedy top-k, w = score * routed_scaling_factor
//   P1 routed gate+up, FP8 block-scaled weights, SiLU(g) * u
//   P2 routed down, times the routing weight w
//   Q1/Q2 shared experts (fused into one MLP of width n_shared * moe_inter)
//   R  combine: h = shared_out + sum of routed (+ residual when one is given)
// The FP8 activation quantisation (one power-of-two scale per token and 128
// channels) is the reading taken here of the pages' FP8 block-scaled expert GEMMs
// (README "Results") and of the quantisation of the experts' inputs to MXFP8 (the
// DeepSeek-V4.1 Flash lecture, "Rounds 12-15" table); the scale form follows the pages' quantiser with
// UE8M0 (power-of-two) scale factors (README "Layout", quant/fp8_block_quant.py).
//
// Parity pins (tests/test_oracle_*.py) tie every function below to something other
// than itself: the OCP E4M3 definition and torch's float8 conversion, closed forms,
// brute-force enumeration, and fp64 library matmuls. The choice of activation
// quantisation (on, power-of-two scale) is a reading of the pages, not something
// the pages print a number for: that choice itself is parity unpinned.
//
// Build: g++ -std=c++17 -O3 -fopenmp -shared -fPIC moe_oracle.cpp -o libmoe_oracle.so
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

typedef struct {
    int32_t hidden;      // H
    int32_t moe_inter;   // I, width of one routed expert
    int32_t n_routed;    // E
    int32_t n_group;     // G, experts form G contiguous groups of E/G
    int32_t topk_group;  // Gk, groups kept per token
    int32_t top_k;       // k, experts kept per token
    int32_t n_shared;    // S, shared experts fused into one MLP of width S*I
    int32_t act_quant;   // 1: FP8 activation quantisation (the method); 0: off
    double routed_scaling_factor;  // s
} orc_cfg_t;

// ---------------------------------------------------------------- E4M3 format
// OCP FP8 E4M3FN: bit 7 sign, bits 6..3 biased exponent (bias 7), bits 2..0
// mantissa. Exponent field 0 encodes subnormals m/8 * 2^-6. S.1111.111 is NaN;
// there is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.
double orc_e4m3_decode(uint8_t code) {
    const int sign = code >> 7;
    const int e = (code >> 3) & 0xF;
    const int m = code & 0x7;
    if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
    double mag;
    if (e == 0)
        mag = std::ldexp((double)m / 8.0, -6);
    else
        mag = std::ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

// Round to the nearest E4M3 value, ties to the even code (the code's last bit is
// the mantissa's last bit), saturating to +-448. NaN maps to 0x7F.
uint8_t orc_e4m3_encode(double v) {
    if (std::isnan(v)) return 0x7F;
    const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
    const double a = std::fabs(v);
    // The 127 finite non-negative codes 0x00..0x7E are increasing in value.
    struct Grid {
        double v[127];
        Grid() {
            for (int c = 0; c < 127; ++c) v[c] = orc_e4m3_decode((uint8_t)c);
        }
    };
    static const Grid G;  // thread-safe one-time initialisation
    const double* grid = G.v;
    if (a >= grid[126]) return sign | 0x7E;
    // first code whose value is >= a
    int hi = (int)(std::lower_bound(grid, grid + 127, a) - grid);
    if (grid[hi] == a) return sign | (uint8_t)hi;
    int lo = hi - 1;
    const double dlo = a - grid[lo], dhi = grid[hi] - a;
    int c;
    if (dlo < dhi)
        c = lo;
    else if (dhi < dlo)
        c = hi;
    else
        c = (lo % 2 == 0) ? lo : hi;
    return sign | (uint8_t)c;
}

// ------------------------------------------------------ activation quantisation
// One block of 128 values: scale = the smallest power of two 2^k with
// amax <= 448 * 2^k (amax = 0 gives scale 1 and all-zero codes), then
// q = RNE-to-E4M3(v / scale). v / scale is exact because the scale is 2^k.
void orc_quant_block(const double* v, int n, uint8_t* q, double* scale_out) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(v[i]));
    double scale = 1.0;
    if (amax > 0.0) {
        int k = (int)std::ceil(std::log2(amax / 448.0));
        while (amax > 448.0 * std::ldexp(1.0, k)) ++k;
        while (amax <= 448.0 * std::ldexp(1.0, k - 1)) --k;
        scale = std::ldexp(1.0, k);
    }
    for (int i = 0; i < n; ++i) q[i] = (amax > 0.0) ? orc_e4m3_encode(v[i] / scale) : 0;
    *scale_out = scale;
}

// Quantise a length-n vector (n a multiple of 128) block by block, and write the
// dequantised values q * scale to vhat (the operand the FP8 GEMM actually sees).
static void quant_dequant(const double* v, int n, double* vhat, uint8_t* q, double* s) {
    for (int b = 0; b < n / 128; ++b) {
        orc_quant_block(v + b * 128, 128, q + b * 128, s + b);
        for (int i = 0; i < 128; ++i) vhat[b * 128 + i] = orc_e4m3_decode(q[b * 128 + i]) * s[b];
    }
}

void orc_quant_rows(const double* v, int rows, int n, uint8_t* q, double* s) {
    std::vector<double> tmp(n);
    for (int r = 0; r < rows; ++r)
        quant_dequant(v + (size_t)r * n, n, tmp.data(), q + (size_t)r * n, s + (size_t)r * (n / 128));
}

static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// -------------------------------------------------------------- bf16 rounding
// Round v to the nearest bf16 value (8 significant bits, exponent range of fp32),
// ties to the even significand, in one step from the double (no detour through
// float, which would round twice). Values at or beyond the overflow threshold give
// infinity, NaN gives the canonical quiet NaN 0x7FC0.
static uint16_t round_bf16(double v) {
    if (std::isnan(v)) return 0x7FC0;
    const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
    const double a = std::fabs(v);
    if (a == 0.0) return sign;
    int e = 0;
    std::frexp(a, &e);       // a in [2^(e-1), 2^e)
    int lead = e - 1;        // exponent of the leading bit
    if (lead < -126) lead = -126;  // subnormals share the smallest normal binade's spacing
    const double quantum = std::ldexp(1.0, lead - 7);  // distance between neighbours here
    const double r = std::nearbyint(a / quantum) * quantum;  // a / quantum is exact
    if (r >= std::ldexp(1.0, 128)) return sign | 0x7F80;
    const float f = (float)r;  // exact: r has at most 8 significant bits
    uint32_t bits;
    std::memcpy(&bits, &f, 4);
    return sign | (uint16_t)(bits >> 16);
}

void orc_round_bf16(const double* v, int n, uint16_t* out) {
    for (int i = 0; i < n; ++i) out[i] = round_bf16(v[i]);
}

// ------------------------------------------------------------------ M: RMSNorm
// Stage M in front of the router (DSV2-236B-MegaKernel stage flowchart, MoE
// subgraph: the hidden state normalised and scaled by its gamma): per token row,
//   x[h] = h[h] / sqrt(mean over the row of h^2 + eps) * gamma[h],
// computed in fp64 and rounded once to bf16. x_exact (optional) receives the value
// before that rounding.
void orc_rmsnorm(const uint16_t* h_bf16, int T, int H, const uint16_t* gamma_bf16, double eps,
                 uint16_t* x_bf16, double* x_exact) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const uint16_t* row = h_bf16 + (size_t)t * H;
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            const double v = bf16_to_double(row[h]);
            ss += v * v;
        }
        const double rms = std::sqrt(ss / H + eps);
        for (int h = 0; h < H; ++h) {
            const double v = bf16_to_double(row[h]) / rms * bf16_to_double(gamma_bf16[h]);
            if (x_exact) x_exact[(size_t)t * H + h] = v;
            x_bf16[(size_t)t * H + h] = round_bf16(v);
        }
    }
}

// ------------------------------------------------------------------ N: router
// logits[t][e] = sum_h x[t][h] * W_router[e][h]  (+ bias[e] when given)
void orc_router_logits(const orc_cfg_t* c, const uint16_t* x_bf16, int T, const float* w_router,
                       const float* bias, double* logits) {
    const int H = c->hidden, E = c->n_routed;
#pragma omp parallel for collapse(2) schedule(static)
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += bf16_to_double(x_bf16[(size_t)t * H + h]) * (double)w_router[(size_t)e * H + h];
            if (bias) acc += (double)bias[e];
            logits[(size_t)t * E + e] = acc;
        }
}

// ------------------------------------------- O: softmax + group-limited top-k
// p = softmax over all E experts. Group j holds experts [j*E/G, (j+1)*E/G) and
// scores max(p) over its members. The topk_group best groups are kept (ties: lower
// group index), the top_k best experts among them are selected (ties: lower expert
// index), listed by score descending then index ascending, and weighted
// w = p * routed_scaling_factor with no renormalisation.
// margin[t] = smallest gap, in probability units, that decided token t: between
// the last kept and first dropped group, between the last selected and first
// unselected eligible expert, and between adjacent selected experts.
void orc_topk(const orc_cfg_t* c, const double* logits, int T, int32_t* ids, double* w,
              double* probs_out, double* margin) {
    const int E = c->n_routed, G = c->n_group, Gk = c->topk_group, k = c->top_k;
    const int per = E / G;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const double* l = logits + (size_t)t * E;
        std::vector<double> p(E);
        double mx = -std::numeric_limits<double>::infinity();
        for (int e = 0; e < E; ++e) mx = std::max(mx, l[e]);
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] = std::exp(l[e] - mx);
            z += p[e];
        }
        for (int e = 0; e < E; ++e) p[e] /= z;
        if (probs_out)
            for (int e = 0; e < E; ++e) probs_out[(size_t)t * E + e] = p[e];

        std::vector<double> gs(G);
        for (int g = 0; g < G; ++g) {
            double m = p[g * per];
            for (int i = 1; i < per; ++i) m = std::max(m, p[g * per + i]);
            gs[g] = m;
        }
        std::vector<int> gord(G);
        for (int g = 0; g < G; ++g) gord[g] = g;
        std::stable_sort(gord.begin(), gord.end(), [&](int a, int b) { return gs[a] > gs[b]; });

        std::vector<int> cand;
        for (int r = 0; r < Gk; ++r)
            for (int i = 0; i < per; ++i) cand.push_back(gord[r] * per + i);
        std::sort(cand.begin(), cand.end());
        std::stable_sort(cand.begin(), cand.end(), [&](int a, int b) { return p[a] > p[b]; });

        double mg = std::numeric_limits<double>::infinity();
        if (Gk < G) mg = std::min(mg, gs[gord[Gk - 1]] - gs[gord[Gk]]);
        if (k < (int)cand.size()) mg = std::min(mg, p[cand[k - 1]] - p[cand[k]]);
        for (int j = 0; j + 1 < k; ++j) mg = std::min(mg, p[cand[j]] - p[cand[j + 1]]);
        if (margin) margin[t] = mg;

        for (int j = 0; j < k; ++j) {
            ids[(size_t)t * k + j] = cand[j];
            w[(size_t)t * k + j] = p[cand[j]] * c->routed_scaling_factor;
        }
    }
}

// ------------------------------------------------------------- permutation
// Stable counting sort of the T*k (token, slot) pairs by expert id. The pair
// (t, j) has flat index f = t*k + j; pairs of one expert keep ascending f.
//   expert_offsets[e] = number of pairs routed to experts < e  (E+1 entries)
//   perm_src[pos]     = f of the pair at permuted position pos
//   inv_pos[f]        = permuted position of pair f
void orc_permute(const orc_cfg_t* c, const int32_t* ids, int T, int32_t* expert_offsets,
                 int32_t* perm_src, int32_t* inv_pos) {
    const int E = c->n_routed, k = c->top_k;
    const int n = T * k;
    std::vector<int32_t> count(E, 0);
    for (int f = 0; f < n; ++f) count[ids[f]]++;
    expert_offsets[0] = 0;
    for (int e = 0; e < E; ++e) expert_offsets[e + 1] = expert_offsets[e] + count[e];
    std::vector<int32_t> next(expert_offsets, expert_offsets + E);
    for (int f = 0; f < n; ++f) {
        const int pos = next[ids[f]]++;
        perm_src[pos] = f;
        inv_pos[f] = pos;
    }
}

// ------------------------------------------------------- P1/P2: one expert MLP
// For one token's dequantised activation xhat[H] and one expert's weights:
//   g = Wg . xhat, u = Wu . xhat           (Wg, Wu: [N, H], block scales [N/128, H/128])
//   a = SiLU(g) * u = g / (1 + e^-g) * u
//   ahat = a, or its FP8 quantise-dequantise when act_quant is on
//   y = w * (Wd . ahat)                    (Wd: [H, N], block scales [H/128, N/128])
// with every weight dequantised as W[o][i] = dec(code[o][i]) * scale[o/128][i/128].
// Writes y[H] (accumulated into y when accumulate != 0).
static void expert_mlp(const double* dec_tab, int H, int N, int act_quant, const double* xhat,
                       const uint8_t* wg, const float* sg, const uint8_t* wu, const float* su,
                       const uint8_t* wd, const float* sd, double w, double* y, int accumulate,
                       double* a_out) {
    const int Hb = H / 128, Nb = N / 128;
    std::vector<double> a(N);
    for (int o = 0; o < N; ++o) {
        double g = 0.0, u = 0.0;
        const uint8_t* rg = wg + (size_t)o * H;
        const uint8_t* ru = wu + (size_t)o * H;
        for (int i = 0; i < H; ++i) {
            g += dec_tab[rg[i]] * (double)sg[(size_t)(o / 128) * Hb + i / 128] * xhat[i];
            u += dec_tab[ru[i]] * (double)su[(size_t)(o / 128) * Hb + i / 128] * xhat[i];
        }
        a[o] = g / (1.0 + std::exp(-g)) * u;
    }
    std::vector<double> ahat(N);
    if (act_quant) {
        std::vector<uint8_t> q(N);
        std::vector<double> s(Nb);
        quant_dequant(a.data(), N, ahat.data(), q.data(), s.data());
    } else {
        ahat = a;
    }
    if (a_out)
        for (int o = 0; o < N; ++o) a_out[o] = ahat[o];
    for (int o = 0; o < H; ++o) {
        const uint8_t* rd = wd + (size_t)o * N;
        double acc = 0.0;
        for (int i = 0; i < N; ++i)
            acc += dec_tab[rd[i]] * (double)sd[(size_t)(o / 128) * Nb + i / 128] * ahat[i];
        y[o] = (accumulate ? y[o] : 0.0) + w * acc;
    }
}

static void make_dec_tab(double* tab) {
    for (int c = 0; c < 256; ++c) tab[c] = orc_e4m3_decode((uint8_t)c);
}

// The activation the expert GEMMs see for token row x: its FP8 quantise-dequantise
// (act_quant on) or the bf16 value itself.
static void token_xhat(const orc_cfg_t* c, const uint16_t* xrow, double* xhat) {
    const int H = c->hidden;
    std::vector<double> xv(H);
    for (int h = 0; h < H; ++h) xv[h] = bf16_to_double(xrow[h]);
    if (c->act_quant) {
        std::vector<uint8_t> q(H);
        std::vector<double> s(H / 128);
        quant_dequant(xv.data(), H, xhat, q.data(), s.data());
    } else {
        for (int h = 0; h < H; ++h) xhat[h] = xv[h];
    }
}

typedef struct {
    const uint8_t *w_gate, *w_up, *w_down;   // [E,I,H], [E,I,H], [E,H,I] E4M3 codes
    const float *s_gate, *s_up, *s_down;     // [E,I/128,H/128], same, [E,H/128,I/128]
    const uint8_t *ws_gate, *ws_up, *ws_down;  // shared [Is,H], [Is,H], [H,Is]; NULL if S=0
    const float *ss_gate, *ss_up, *ss_down;    // [Is/128,H/128], same, [H/128,Is/128]
} orc_weights_t;

// One routed (token, expert, weight) row: y[H] = w * expert_e(xhat(token)).
// Also writes the expert's (dequantised) intermediate activation to a_out[I] if given.
void orc_expert_row(const orc_cfg_t* c, const orc_weights_t* W, const uint16_t* x_row, int expert,
                    double w, double* y, double* a_out) {
    const int H = c->hidden, I = c->moe_inter, Hb = H / 128, Ib = I / 128;
    double tab[256];
    make_dec_tab(tab);
    std::vector<double> xhat(H);
    token_xhat(c, x_row, xhat.data());
    const size_t e = (size_t)expert;
    expert_mlp(tab, H, I, c->act_quant, xhat.data(), W->w_gate + e * I * H, W->s_gate + e * Ib * Hb,
               W->w_up + e * I * H, W->s_up + e * Ib * Hb, W->w_down + e * H * I,
               W->s_down + e * Hb * Ib, w, y, 0, a_out);
}

// The shared experts for one token: y[H] = shared_MLP(xhat(token)), weight 1.
void orc_shared_row(const orc_cfg_t* c, const orc_weights_t* W, const uint16_t* x_row, double* y) {
    const int H = c->hidden, Is = c->n_shared * c->moe_inter;
    double tab[256];
    make_dec_tab(tab);
    std::vector<double> xhat(H);
    token_xhat(c, x_row, xhat.data());
    if (c->n_shared == 0) {
        for (int h = 0; h < H; ++h) y[h] = 0.0;
        return;
    }
    expert_mlp(tab, H, Is, c->act_quant, xhat.data(), W->ws_gate, W->ss_gate, W->ws_up, W->ss_up,
               W->ws_down, W->ss_down, 1.0, y, 0, nullptr);
}

// R: the layer output for the listed tokens, in fp64.
//   out[i][:] = sum_j w[t][j] * expert_{ids[t][j]}(xhat_t) + shared(xhat_t) (+ residual[t])
// for t = tokens[i]. ids / w are the routing of all T tokens ([T,k], from orc_topk
// or given by the caller); residual is bf16 [T,H] or NULL.
void orc_forward_tokens(const orc_cfg_t* c, const orc_weights_t* W, const uint16_t* x_bf16,
                        const int32_t* ids, const double* w, const uint16_t* residual_bf16,
                        const int32_t* tokens, int n_tokens, double* out) {
    const int H = c->hidden, I = c->moe_inter, k = c->top_k, Hb = H / 128, Ib = I / 128;
    const int Is = c->n_shared * I;
    double tab[256];
    make_dec_tab(tab);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n_tokens; ++i) {
        const int t = tokens[i];
        std::vector<double> xhat(H);
        token_xhat(c, x_bf16 + (size_t)t * H, xhat.data());
        double* o = out + (size_t)i * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            const size_t e = (size_t)ids[(size_t)t * k + j];
            expert_mlp(tab, H, I, c->act_quant, xhat.data(), W->w_gate + e * I * H,
                       W->s_gate + e * Ib * Hb, W->w_up + e * I * H, W->s_up + e * Ib * Hb,
                       W->w_down + e * H * I, W->s_down + e * Hb * Ib, w[(size_t)t * k + j], o, 1,
                       nullptr);
        }
        if (c->n_shared > 0)
            expert_mlp(tab, H, Is, c->act_quant, xhat.data(), W->ws_gate, W->ss_gate, W->ws_up,
                       W->ss_up, W->ws_down, W->ss_down, 1.0, o, 1, nullptr);
        if (residual_bf16)
            for (int h = 0; h < H; ++h) o[h] += bf16_to_double(residual_bf16[(size_t)t * H + h]);
    }
}

// ------------------------------------------------------------------ MXFP8
// The MXFP8 variant of the expert MLPs: E4M3 codes with one UE8M0 (power-of-two)
// scale per 32 consecutive values along K, for the weights (per output row) and the
// activations (per token) alike (Mixture-of-Kittens Table 2, its MXFP8 routed-expert
// rows; the DeepSeek-V4.1 Flash lecture's conversion of the weights' block scales to
// the MX layout at load time and its MXFP8 quantisation of the experts' inputs,
// "Round 1->2" and "Rounds 12-15").
// An E8M0 byte b encodes 2^(b-127); 0xFF is NaN.
double orc_e8m0_decode(uint8_t b) {
    if (b == 0xFF) return std::numeric_limits<double>::quiet_NaN();
    return std::ldexp(1.0, (int)b - 127);
}

// One block of 32 values: the scale rule of orc_quant_block (the smallest 2^k with
// amax <= 448 * 2^k; amax = 0 gives 2^0), with k kept >= -126 (a block whose amax is
// below 448 * 2^-127 still gets 2^-126), stored as the byte k + 127.
static void quant_block_mx(const double* v, uint8_t* q, uint8_t* s) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
    int k = 0;
    if (amax > 0.0) {
        k = (int)std::ceil(std::log2(amax / 448.0));
        while (amax > 448.0 * std::ldexp(1.0, k)) ++k;
        while (amax <= 448.0 * std::ldexp(1.0, k - 1)) --k;
        if (k < -126) k = -126;
    }
    const double scale = std::ldexp(1.0, k);
    for (int i = 0; i < 32; ++i) q[i] = (amax > 0.0) ? orc_e4m3_encode(v[i] / scale) : 0;
    *s = (uint8_t)(k + 127);
}

// Rows of n values (n a multiple of 32) -> codes [rows, n] and E8M0 scales [rows, n/32].
void orc_quant_rows_mx(const double* v, int rows, int n, uint8_t* q, uint8_t* s) {
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < n / 32; ++b)
            quant_block_mx(v + (size_t)r * n + b * 32, q + (size_t)r * n + b * 32, s + (size_t)r * (n / 32) + b);
}

static void quant_dequant_mx(const double* v, int n, double* vhat) {
    uint8_t q[32], s;
    for (int b = 0; b < n / 32; ++b) {
        quant_block_mx(v + b * 32, q, &s);
        for (int i = 0; i < 32; ++i) vhat[b * 32 + i] = orc_e4m3_decode(q[i]) * orc_e8m0_decode(s);
    }
}

// One MXFP8 expert MLP (the steps of expert_mlp with per-32 E8M0 scales):
//   W[o][i] = dec(code[o][i]) * 2^(s[o][i/32] - 127)   for Wg, Wu [N, H] and Wd [H, N]
//   g = Wg . xhat, u = Wu . xhat, a = SiLU(g) * u, ahat = MX quantise-dequantise of a,
//   y (+)= w * (Wd . ahat)
static void expert_mlp_mx(const double* dec_tab, int H, int N, int act_quant, const double* xhat,
                          const uint8_t* wg, const uint8_t* sg, const uint8_t* wu, const uint8_t* su,
                          const uint8_t* wd, const uint8_t* sd, double w, double* y, int accumulate) {
    const int H32 = H / 32, N32 = N / 32;
    std::vector<double> a(N), ahat(N);
    for (int o = 0; o < N; ++o) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < H; ++i) {
            g += dec_tab[wg[(size_t)o * H + i]] * orc_e8m0_decode(sg[(size_t)o * H32 + i / 32]) * xhat[i];
            u += dec_tab[wu[(size_t)o * H + i]] * orc_e8m0_decode(su[(size_t)o * H32 + i / 32]) * xhat[i];
        }
        a[o] = g / (1.0 + std::exp(-g)) * u;
    }
    if (act_quant)
        quant_dequant_mx(a.data(), N, ahat.data());
    else
        ahat = a;
    for (int o = 0; o < H; ++o) {
        double acc = 0.0;
        for (int i = 0; i < N; ++i)
            acc += dec_tab[wd[(size_t)o * N + i]] * orc_e8m0_decode(sd[(size_t)o * N32 + i / 32]) * ahat[i];
        y[o] = (accumulate ? y[o] : 0.0) + w * acc;
    }
}

typedef struct {
    const uint8_t *w_gate, *w_up, *w_down;     // E4M3 codes, layouts as orc_weights_t
    const uint8_t *s_gate, *s_up, *s_down;     // E8M0 [E,I,H/32], [E,I,H/32], [E,H,I/32]
    const uint8_t *ws_gate, *ws_up, *ws_down;  // shared codes [Is,H], [Is,H], [H,Is]
    const uint8_t *ss_gate, *ss_up, *ss_down;  // E8M0 [Is,H/32], [Is,H/32], [H,Is/32]
} orc_weights_mx_t;

// R with MXFP8 experts, for the listed tokens (as orc_forward_tokens):
//   out[i] = sum_j w[t][j] * expert_mx_{ids[t][j]}(xhat_t) + shared_mx(xhat_t) (+ residual[t])
// where xhat_t is the MX quantise-dequantise of the bf16 row (act_quant on).
void orc_forward_tokens_mx(const orc_cfg_t* c, const orc_weights_mx_t* W, const uint16_t* x_bf16,
                           const int32_t* ids, const double* w, const uint16_t* residual_bf16,
                           const int32_t* tokens, int n_tokens, double* out) {
    const int H = c->hidden, I = c->moe_inter, k = c->top_k;
    const int Is = c->n_shared * I;
    double tab[256];
    make_dec_tab(tab);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n_tokens; ++i) {
        const int t = tokens[i];
        std::vector<double> xv(H), xhat(H);
        for (int h = 0; h < H; ++h) xv[h] = bf16_to_double(x_bf16[(size_t)t * H + h]);
        if (c->act_quant)
            quant_dequant_mx(xv.data(), H, xhat.data());
        else
            xhat = xv;
        double* o = out + (size_t)i * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            const size_t e = (size_t)ids[(size_t)t * k + j];
            expert_mlp_mx(tab, H, I, c->act_quant, xhat.data(), W->w_gate + e * I * H,
                          W->s_gate + e * I * (H / 32), W->w_up + e * I * H, W->s_up + e * I * (H / 32),
                          W->w_down + e * H * I, W->s_down + e * H * (I / 32), w[(size_t)t * k + j], o, 1);
        }
        if (c->n_shared > 0)
            expert_mlp_mx(tab, H, Is, c->act_quant, xhat.data(), W->ws_gate, W->ss_gate, W->ws_up, W->ss_up,
                          W->ws_down, W->ss_down, 1.0, o, 1);
        if (residual_bf16)
            for (int h = 0; h < H; ++h) o[h] += bf16_to_double(residual_bf16[(size_t)t * H + h]);
    }
}

// ---------------------------------------------------------------- backward
// The layer's backward for an output gradient dout[T][H]: the training workload of the
// Mixture-of-Kittens page (Table 1's backward columns; the abstract's training of the
// expert MLPs), for one layer on one device. The forward's expert choice (ids) is held
// fixed: selection is piecewise constant in the inputs, so gradients reach the router
// only through the routing weights of the kept experts, w = s * p_e.
// Reading taken here (the pages give no formulas): the FP8 quantisers are
// straight-through (the derivative of x -> xhat and of a -> ahat is taken as 1), the
// weights are their dequantised FP8 values, and the forward values g, u, a, ahat are
// those the forward computes (FP8 activations when act_quant is on). Per routed pair
// (t, j) with expert e:
//   z   = Wd_e . ahat                    (expert output before weighting)
//   dw  = <dout_t, z>
//   da  = w * Wd_e^T dout_t
//   dg  = da * u * sig(g) * (1 + g * (1 - sig(g)))      (d/dg of g * sig(g), times u)
//   du  = da * g * sig(g)
//   dx_t  += Wg_e^T dg + Wu_e^T du
//   dWd_e += (w * dout_t) (x) ahat,  dWg_e += dg (x) xhat_t,  dWu_e += du (x) xhat_t
// The shared experts: the same with w = 1 and no routing term. The router
// (logits = Wr . x + bias on the unquantised input x):
//   dp_e = s * dw for the kept experts of the token, 0 for the others
//   dlogit = p * (dp - <p, dp>)                       (softmax over all E)
//   dx_t += Wr^T dlogit,  dWr += dlogit (x) x_t,  dbias += dlogit
// Inputs and outputs are fp64 here so that finite differences can probe the function;
// x is the layer input (bf16 values widened), w_router / bias fp64 copies.
// The forward used by those finite differences (fixed ids, w recomputed from x):
//   out_t = sum_j s * p_{e_j}(x_t) * z_{e_j}(xhat_t) + shared(xhat_t)
void orc_forward_fixed_ids_d(const orc_cfg_t* c, const orc_weights_t* W, const double* w_router,
                             const double* bias, const double* x, int T, const int32_t* ids, double* out) {
    const int H = c->hidden, I = c->moe_inter, E = c->n_routed, k = c->top_k, Hb = H / 128, Ib = I / 128;
    const int Is = c->n_shared * I;
    double tab[256];
    make_dec_tab(tab);
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        const double* xt = x + (size_t)t * H;
        std::vector<double> xhat(H), l(E);
        if (c->act_quant) {
            std::vector<uint8_t> q(H);
            std::vector<double> sc(H / 128);
            quant_dequant(xt, H, xhat.data(), q.data(), sc.data());
        } else {
            for (int h = 0; h < H; ++h) xhat[h] = xt[h];
        }
        double mx = -std::numeric_limits<double>::infinity();
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h) acc += xt[h] * w_router[(size_t)e * H + h];
            l[e] = acc + (bias ? bias[e] : 0.0);
            mx = std::max(mx, l[e]);
        }
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += std::exp(l[e] - mx);
        double* o = out + (size_t)t * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            const size_t e = (size_t)ids[(size_t)t * k + j];
            const double w = c->routed_scaling_factor * std::exp(l[e] - mx) / z;
            expert_mlp(tab, H, I, c->act_quant, xhat.data(), W->w_gate + e * I * H, W->s_gate + e * Ib * Hb,
                       W->w_up + e * I * H, W->s_up + e * Ib * Hb, W->w_down + e * H * I,
                       W->s_down + e * Hb * Ib, w, o, 1, nullptr);
        }
        if (c->n_shared > 0)
            expert_mlp(tab, H, Is, c->act_quant, xhat.data(), W->ws_gate, W->ss_gate, W->ws_up, W->ss_up,
                       W->ws_down, W->ss_down, 1.0, o, 1, nullptr);
    }
}

// One expert MLP's backward for one token. Adds to dx[H] and, through the callback
// arrays, hands back the per-row vectors the weight gradients need:
//   ahat[N], dg[N], du[N]; returns dw = <dout, Wd . ahat>.
static double expert_mlp_bwd(const double* dec_tab, int H, int N, int act_quant, const double* xhat,
                             const uint8_t* wg, const float* sg, const uint8_t* wu, const float* su,
                             const uint8_t* wd, const float* sd, double w, const double* dout, double* dx,
                             double* ahat_out, double* dg_out, double* du_out) {
    const int Hb = H / 128, Nb = N / 128;
    std::vector<double> g(N), u(N), a(N), ahat(N);
    for (int o = 0; o < N; ++o) {
        double gg = 0.0, uu = 0.0;
        for (int i = 0; i < H; ++i) {
            gg += dec_tab[wg[(size_t)o * H + i]] * (double)sg[(size_t)(o / 128) * Hb + i / 128] * xhat[i];
            uu += dec_tab[wu[(size_t)o * H + i]] * (double)su[(size_t)(o / 128) * Hb + i / 128] * xhat[i];
        }
        g[o] = gg;
        u[o] = uu;
        a[o] = gg / (1.0 + std::exp(-gg)) * uu;
    }
    if (act_quant) {
        std::vector<uint8_t> q(N);
        std::vector<double> s(Nb);
        quant_dequant(a.data(), N, ahat.data(), q.data(), s.data());
    } else {
        ahat = a;
    }
    // z = Wd . ahat and da = w * Wd^T dout, one pass over Wd
    double dw = 0.0;
    std::vector<double> da(N, 0.0);
    for (int o = 0; o < H; ++o) {
        double zo = 0.0;
        for (int i = 0; i < N; ++i) {
            const double wv = dec_tab[wd[(size_t)o * N + i]] * (double)sd[(size_t)(o / 128) * Nb + i / 128];
            zo += wv * ahat[i];
            da[i] += w * wv * dout[o];
        }
        dw += dout[o] * zo;
    }
    std::vector<double> dg(N), du(N);
    for (int o = 0; o < N; ++o) {
        const double sg_ = 1.0 / (1.0 + std::exp(-g[o]));
        dg[o] = da[o] * u[o] * sg_ * (1.0 + g[o] * (1.0 - sg_));
        du[o] = da[o] * g[o] * sg_;
    }
    for (int o = 0; o < N; ++o)
        for (int i = 0; i < H; ++i) {
            const double wgv = dec_tab[wg[(size_t)o * H + i]] * (double)sg[(size_t)(o / 128) * Hb + i / 128];
            const double wuv = dec_tab[wu[(size_t)o * H + i]] * (double)su[(size_t)(o / 128) * Hb + i / 128];
            dx[i] += wgv * dg[o] + wuv * du[o];
        }
    for (int o = 0; o < N; ++o) {
        ahat_out[o] = ahat[o];
        dg_out[o] = dg[o];
        du_out[o] = du[o];
    }
    return dw;
}

// Gradients of L = sum_t <dout_t, out_t>: dx [T,H]; dwg, dwu [E,I,H]; dwd [E,H,I];
// dwsg, dwsu [Is,H], dwsd [H,Is] (ignored when S = 0); dwr [E,H]; dbias [E]. The
// weight-gradient outputs may be NULL (dwg: the routed ones; dwsg: the shared ones;
// dwr: the router's): dx_t depends on token t alone, so dx of a sample of tokens is
// exact when only their rows are passed.
// w [T,k] are the routing weights the forward applied (s * p of the kept experts).
void orc_backward_d(const orc_cfg_t* c, const orc_weights_t* W, const double* w_router, const double* bias,
                    const double* x, int T, const int32_t* ids, const double* w, const double* dout, double* dx,
                    double* dwg, double* dwu, double* dwd, double* dwsg, double* dwsu, double* dwsd, double* dwr,
                    double* dbias) {
    const int H = c->hidden, I = c->moe_inter, E = c->n_routed, k = c->top_k, Hb = H / 128, Ib = I / 128;
    const int Is = c->n_shared * I;
    const double s = c->routed_scaling_factor;
    double tab[256];
    make_dec_tab(tab);
    // per pair (t, j): ahat, dg, du; per token: xhat and the router gradient dlogit
    std::vector<double> p_ahat((size_t)T * k * I), p_dg((size_t)T * k * I), p_du((size_t)T * k * I);
    std::vector<double> xhat_all((size_t)T * H), dlogit((size_t)T * E);
    std::vector<double> s_ahat((size_t)T * Is), s_dg((size_t)T * Is), s_du((size_t)T * Is);
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        const double* xt = x + (size_t)t * H;
        double* xhat = xhat_all.data() + (size_t)t * H;
        if (c->act_quant) {
            std::vector<uint8_t> q(H);
            std::vector<double> sc(H / 128);
            quant_dequant(xt, H, xhat, q.data(), sc.data());
        } else {
            for (int h = 0; h < H; ++h) xhat[h] = xt[h];
        }
        const double* dt = dout + (size_t)t * H;
        double* dxt = dx + (size_t)t * H;
        for (int h = 0; h < H; ++h) dxt[h] = 0.0;
        std::vector<double> dp(E, 0.0);
        for (int j = 0; j < k; ++j) {
            const size_t f = (size_t)t * k + j, e = (size_t)ids[f];
            const double dwj = expert_mlp_bwd(
                tab, H, I, c->act_quant, xhat, W->w_gate + e * I * H, W->s_gate + e * Ib * Hb, W->w_up + e * I * H,
                W->s_up + e * Ib * Hb, W->w_down + e * H * I, W->s_down + e * Hb * Ib, w[f], dt, dxt,
                p_ahat.data() + f * I, p_dg.data() + f * I, p_du.data() + f * I);
            dp[e] += s * dwj;
        }
        if (c->n_shared > 0)
            expert_mlp_bwd(tab, H, Is, c->act_quant, xhat, W->ws_gate, W->ss_gate, W->ws_up, W->ss_up, W->ws_down,
                           W->ss_down, 1.0, dt, dxt, s_ahat.data() + (size_t)t * Is, s_dg.data() + (size_t)t * Is,
                           s_du.data() + (size_t)t * Is);
        // router: softmax over all E of logits = Wr . x + bias
        std::vector<double> l(E), p(E);
        double mx = -std::numeric_limits<double>::infinity();
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h) acc += xt[h] * w_router[(size_t)e * H + h];
            l[e] = acc + (bias ? bias[e] : 0.0);
            mx = std::max(mx, l[e]);
        }
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += (p[e] = std::exp(l[e] - mx));
        double pdp = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] /= z;
            pdp += p[e] * dp[e];
        }
        for (int e = 0; e < E; ++e) {
            const double dl = p[e] * (dp[e] - pdp);
            dlogit[(size_t)t * E + e] = dl;
            for (int h = 0; h < H; ++h) dxt[h] += w_router[(size_t)e * H + h] * dl;
        }
    }
    // weight gradients: sums over the token pairs of each expert, in token order
    // (NULL outputs are skipped: dx alone is exact for any subset of tokens)
#pragma omp parallel for schedule(dynamic, 1)
    for (int e = 0; e < (dwg ? E : 0); ++e) {
        double* gW = dwg + (size_t)e * I * H;
        double* uW = dwu + (size_t)e * I * H;
        double* dW = dwd + (size_t)e * H * I;
        std::fill(gW, gW + (size_t)I * H, 0.0);
        std::fill(uW, uW + (size_t)I * H, 0.0);
        std::fill(dW, dW + (size_t)H * I, 0.0);
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j) {
                const size_t f = (size_t)t * k + j;
                if (ids[f] != e) continue;
                const double* xh = xhat_all.data() + (size_t)t * H;
                const double* dt = dout + (size_t)t * H;
                const double* ah = p_ahat.data() + f * I;
                const double* dg = p_dg.data() + f * I;
                const double* du = p_du.data() + f * I;
                for (int o = 0; o < I; ++o)
                    for (int i = 0; i < H; ++i) {
                        gW[(size_t)o * H + i] += dg[o] * xh[i];
                        uW[(size_t)o * H + i] += du[o] * xh[i];
                    }
                for (int o = 0; o < H; ++o)
                    for (int i = 0; i < I; ++i) dW[(size_t)o * I + i] += w[f] * dt[o] * ah[i];
            }
    }
#pragma omp parallel for schedule(static)
    for (int e = 0; e < (dwr ? E : 0); ++e) {
        double* rW = dwr + (size_t)e * H;
        std::fill(rW, rW + H, 0.0);
        double db = 0.0;
        for (int t = 0; t < T; ++t) {
            const double dl = dlogit[(size_t)t * E + e];
            db += dl;
            for (int h = 0; h < H; ++h) rW[h] += dl * x[(size_t)t * H + h];
        }
        if (dbias) dbias[e] = db;
    }
    if (c->n_shared > 0 && dwsg) {
#pragma omp parallel for schedule(static)
        for (int o = 0; o < Is; ++o) {
            for (int i = 0; i < H; ++i) {
                double ag = 0.0, au = 0.0;
                for (int t = 0; t < T; ++t) {
                    ag += s_dg[(size_t)t * Is + o] * xhat_all[(size_t)t * H + i];
                    au += s_du[(size_t)t * Is + o] * xhat_all[(size_t)t * H + i];
                }
                dwsg[(size_t)o * H + i] = ag;
                dwsu[(size_t)o * H + i] = au;
            }
        }
#pragma omp parallel for schedule(static)
        for (int o = 0; o < H; ++o)
            for (int i = 0; i < Is; ++i) {
                double acc = 0.0;
                for (int t = 0; t < T; ++t) acc += dout[(size_t)t * H + o] * s_ahat[(size_t)t * Is + i];
                dwsd[(size_t)o * Is + i] = acc;
            }
    }
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

}  // extern "C"

// MoE expert-layer oracle: plain, slow, fp64 CPU implementation.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load or call this
// library; only the test suite, the smoke check and the benchmark's CPU-baseline
// leg do.  It shares no code, header or constant with the CUDA implementation.
//
// What it computes (sources, by page title and section):
//  * "DeepSeek-V4 并行策略：重叠计算与通信" (blog.lpkt.cn), section "EP 对 IB 网络的优化":
//    an MoE layer is Dispatch -> Expert Compute -> Combine.
//  * DeepSeek-V4 report reading (10100.com), section on fine-grained overlap of the EP
//    all-to-all: the expert stage is Linear + activation + Linear.
//  * DeepSeek-V4 report, Thai translation (itsolotime.com), section 1.4 "observations and
//    suggestions": each token-expert pair costs 6hd FLOP covering the SwiGLU gate
//    projection, the up projection and the down projection; the combine payload is BF16.
//  * The same page, section 1.4, bullet on the compute-to-bandwidth ratio: the dispatch
//    payload is FP8 (the combine payload BF16).
//  * The same page, section 1.4, bullet on the activation function: a cheap element-wise
//    activation without exponentials or divisions in place of SwiGLU, with the gating
//    projection removed (the parameter budget then allows a wider intermediate).
//  * The same page, section 3, and the 10100.com reading, section on batch-invariant and
//    deterministic kernels: results must not depend on batch size or run.
//
// Readings taken where the pages are silent (each repeated next to the code below):
//  * router: top-k over fp32 logits, ties go to the lower expert index; the gate is the
//    softmax over the k selected logits.
//  * stable permute: permuted rows are ordered by (expert, token).
//  * SwiGLU: h = silu(x W1) * (x W3), silu(a) = a / (1 + exp(-a)); h is rounded to bf16
//    (round to nearest, ties to even) before the down projection when round_h != 0.
//  * expert output rows: with round_h != 0 each row o = h W2 is rounded to bf16 as well (the
//    BF16 combine payload of the report translation, section 1.4), and the combine and the
//    gate gradient read those bf16 rows.
//  * cheap activation (no W3 given): h = relu(x W1)^2, squared ReLU, an element-wise function
//    with neither exponential nor division; h rounded to bf16 as above.
//  * combine: y_t = sum_j g_j * o_j, here in fp64.
//  * FP8 dispatch: each token row is sent as FP8 E4M3 values with one fp32 scale per row,
//    s_t = amax_c |x_tc| / 448 (448 = the largest E4M3 value; s_t = 1 for an all-zero row),
//    q = e4m3(x / s_t) with x / s_t an fp32 division and e4m3() rounding to nearest even
//    with saturation at 448.  The first projections use weights in the same format with one
//    scale per (expert, output column), taken over the input dimension.  The expert then
//    runs on the dequantized values q s, exactly as on bf16 inputs.
//  * backward: the derivative of the bf16 rounding of h is taken as 1; with round_grad the
//    matrix-product operands dO = g dy, da and db are rounded to bf16 (round to nearest
//    even) like h, each product accumulating exactly (fp64).
//  * rounding-flip allowance (a test bound, not part of the layer): both the oracle and an
//    fp32 implementation round h, o, dO, da and db to bf16, but from pre-rounding values that
//    differ by the fp32 implementation's own rounding errors, so an operand whose value lies
//    near a bf16 rounding midpoint may round to the neighbouring bf16 value there.  For each
//    such operand the oracle computes, from its own fp64 values alone, the largest distance
//    between the two roundings, on each side, using a model of fp32 arithmetic (FlipModel
//    below); every gradient element then gets, on top of the stated tolerance, the largest
//    change that those operands can cause together (each operand's signed deviation
//    interval times what multiplies it in the element, summed over the element's terms).
//
// All arithmetic is fp64.  bf16 inputs are passed as their raw 16-bit patterns and
// widened exactly.  Loops run in the plain order of the definitions; OpenMP only
// splits independent tokens, rows or output rows between threads.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <omp.h>

namespace {

inline double widen(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}
inline double widen(double v) { return v; }

// Nearest bf16 value to v, ties to even (bf16: 8 significant bits, float's exponent range).
double round_bf16(double v) {
  if (v == 0.0 || std::isnan(v) || std::isinf(v)) return v;
  const double a = std::fabs(v);
  double r;
  if (a < std::ldexp(1.0, -126)) {
    // subnormal range of bf16: a multiple of 2^-133
    r = std::nearbyint(std::ldexp(a, 133));
    r = std::ldexp(r, -133);
  } else {
    int ex;
    double m = std::frexp(a, &ex);          // a = m * 2^ex, m in [0.5, 1)
    r = std::nearbyint(std::ldexp(m, 8));   // 8 significant bits, ties to even
    r = std::ldexp(r, ex - 8);
    if (r >= std::ldexp(1.0, 128)) r = INFINITY;
  }
  return v < 0 ? -r : r;
}

double sigmoid(double a) { return 1.0 / (1.0 + std::exp(-a)); }

// Nearest FP8 E4M3 value to v (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
// infinities): ties to even; magnitudes above 448, the largest finite value, saturate to it.
double round_e4m3(double v) {
  if (v == 0.0 || std::isnan(v)) return v;
  const double a = std::fabs(v);
  double r;
  if (a < std::ldexp(1.0, -6)) {
    // subnormal range: multiples of 2^-9
    r = std::ldexp(std::nearbyint(std::ldexp(a, 9)), -9);
  } else {
    int ex;
    const double m = std::frexp(a, &ex);  // a = m 2^ex, m in [0.5, 1)
    r = std::ldexp(std::nearbyint(std::ldexp(m, 4)), ex - 4);  // 4 significant bits
  }
  if (r > 448.0) r = 448.0;
  return v < 0 ? -r : r;
}

// fp32 scale of a block whose largest magnitude is amax (an fp32 value): amax / 448 as an
// fp32 division (the double quotient rounded once to float is the correctly rounded fp32
// quotient), 1 for an all-zero block.
double e4m3_scale(double amax) {
  if (amax == 0.0) return 1.0;
  return static_cast<double>(static_cast<float>(amax / 448.0));
}
// x quantized with scale s: e4m3 of the fp32 quotient x / s
double e4m3_quant(double x, double s) {
  return round_e4m3(static_cast<double>(static_cast<float>(x / s)));
}

// Router for one token.  Experts are ordered by (logit descending, index ascending) and
// the first k are kept; the gate is the softmax over those k logits.
void route_token(const double* l, int E, int k, int32_t* idx, double* gate) {
  std::vector<char> taken(E, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      // strict '>' keeps the lower index when two logits compare equal (+0 == -0 too)
      if (best < 0 || l[e] > l[best]) best = e;
    }
    taken[best] = 1;
    idx[j] = best;
  }
  const double m = l[idx[0]];
  double s = 0.0;
  for (int j = 0; j < k; ++j) s += std::exp(l[idx[j]] - m);
  for (int j = 0; j < k; ++j) gate[j] = std::exp(l[idx[j]] - m) / s;
}

// One expert applied to one row x[0..d): a = x W1, b = x W3, h = silu(a) * b, o = h W2;
// without W3 (W3e null) the cheap activation: h = relu(a)^2 (b is left zero).  With round_h,
// h and o are rounded to bf16.  W1e, W3e are [d][dff] and W2e is [dff][d], row-major.
// Optional by-products of ffn_row for the rounding-flip allowance: sa, sb = the sums of the
// squared running partial sums of a and b (in the order the loops below form a and b), and
// vh = h before its bf16 rounding; so, vo = the same for o (null: not traced).
struct FwdTrace {
  double* sa;
  double* sb;
  double* vh;
  double* so = nullptr;
  double* vo = nullptr;
};

template <class V>
void ffn_row(const V* x, const V* W1e, const V* W3e, const V* W2e, int d, int dff, int round_h,
             double* a, double* b, double* h, double* o, const FwdTrace* tr = nullptr) {
  for (int f = 0; f < dff; ++f) { a[f] = 0.0; b[f] = 0.0; }
  if (tr) for (int f = 0; f < dff; ++f) { tr->sa[f] = 0.0; tr->sb[f] = 0.0; }
  for (int c = 0; c < d; ++c) {
    const double xc = widen(x[c]);
    const V* w1 = W1e + static_cast<int64_t>(c) * dff;
    for (int f = 0; f < dff; ++f) a[f] += xc * widen(w1[f]);
    if (tr) for (int f = 0; f < dff; ++f) tr->sa[f] += a[f] * a[f];
    if (W3e) {
      const V* w3 = W3e + static_cast<int64_t>(c) * dff;
      for (int f = 0; f < dff; ++f) b[f] += xc * widen(w3[f]);
      if (tr) for (int f = 0; f < dff; ++f) tr->sb[f] += b[f] * b[f];
    }
  }
  for (int f = 0; f < dff; ++f) {
    double hv;
    if (W3e) {
      hv = a[f] / (1.0 + std::exp(-a[f])) * b[f];
    } else {
      const double r = a[f] > 0.0 ? a[f] : 0.0;
      hv = r * r;
    }
    if (tr) tr->vh[f] = hv;
    h[f] = round_h ? round_bf16(hv) : hv;
  }
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  const bool tro = tr && tr->so;
  if (tro) for (int c = 0; c < d; ++c) tr->so[c] = 0.0;
  for (int f = 0; f < dff; ++f) {
    const V* w2 = W2e + static_cast<int64_t>(f) * d;
    for (int c = 0; c < d; ++c) o[c] += h[f] * widen(w2[c]);
    if (tro) for (int c = 0; c < d; ++c) tr->so[c] += o[c] * o[c];
  }
  for (int c = 0; c < d; ++c) {
    if (tr && tr->vo) tr->vo[c] = o[c];
    if (round_h) o[c] = round_bf16(o[c]);
  }
}

// Backward of one token-expert pair given its forward values (a, b, h, o), its gate g and
// the upstream gradient dy of the layer output:
//   dgate = <o, dy>, dO = g dy, dh = dO W2^T,
//   da = dh * b * silu'(a) with silu'(a) = s (1 + a (1 - s)), s = sigmoid(a),
//   db = dh * silu(a),  dxp = da W1^T + db W3^T;
// without W3: da = dh * 2 relu(a) (the derivative of relu(a)^2), db = 0, dxp = da W1^T.
// With round_grad != 0, dO, da and db are rounded to bf16 where they become operands of a
// matrix product (dh, dxp and the weight gradients), the reading that every product of the
// layer takes bf16 operands and accumulates exactly (here in fp64).
// Optional by-products of ffn_row_bwd for the rounding-flip allowance: sdh = the sums of the
// squared running partial sums of dh; vda, vdb = da and db before their bf16 rounding.
struct BwdTrace {
  double* sdh;
  double* vda;
  double* vdb;
};

template <class V>
void ffn_row_bwd(const V* W1e, const V* W3e, const V* W2e, int d, int dff, double g,
                 const double* dy, const double* a, const double* b, const double* o,
                 int round_grad, double* dgate, double* dO, double* dh, double* da, double* db,
                 double* dxp, const BwdTrace* tr = nullptr) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += o[c] * dy[c];
  *dgate = s;
  for (int c = 0; c < d; ++c) dO[c] = round_grad ? round_bf16(g * dy[c]) : g * dy[c];
  for (int f = 0; f < dff; ++f) {
    const V* w2 = W2e + static_cast<int64_t>(f) * d;
    double acc = 0.0, sq = 0.0;
    for (int c = 0; c < d; ++c) {
      acc += dO[c] * widen(w2[c]);
      if (tr) sq += acc * acc;
    }
    dh[f] = acc;
    if (tr) tr->sdh[f] = sq;
  }
  for (int f = 0; f < dff; ++f) {
    if (W3e) {
      const double sg = sigmoid(a[f]);
      da[f] = dh[f] * b[f] * sg * (1.0 + a[f] * (1.0 - sg));
      db[f] = dh[f] * a[f] * sg;
    } else {
      da[f] = dh[f] * 2.0 * (a[f] > 0.0 ? a[f] : 0.0);
      db[f] = 0.0;
    }
    if (tr) {
      tr->vda[f] = da[f];
      tr->vdb[f] = db[f];
    }
    if (round_grad) {
      da[f] = round_bf16(da[f]);
      db[f] = round_bf16(db[f]);
    }
  }
  for (int c = 0; c < d; ++c) {
    const V* w1 = W1e + static_cast<int64_t>(c) * dff;
    double acc = 0.0;
    if (W3e) {
      const V* w3 = W3e + static_cast<int64_t>(c) * dff;
      for (int f = 0; f < dff; ++f) acc += da[f] * widen(w1[f]) + db[f] * widen(w3[f]);
    } else {
      for (int f = 0; f < dff; ++f) acc += da[f] * widen(w1[f]);
    }
    dxp[c] = acc;
  }
}

// ---------------------------------------------------------- rounding-flip allowance
// Model of the fp32 arithmetic of an implementation that rounds the same operands to bf16
// (the allowance's only parameters):
//  * acc: an fp32 sum s = t_1 + ... + t_n lies within acc * sqrt(sum_j s_j^2) of the exact
//    sum, s_j its running partial sums.  If each addition's rounding error is independent,
//    zero-mean and at most eps relative, the Azuma-Hoeffding inequality bounds the sum's error
//    by lambda * eps * sqrt(sum_j s_j^2) with probability at least 1 - 2 exp(-lambda^2 / 2)
//    (the probabilistic rounding-error analysis of Higham and Mary, SIAM J. Sci. Comput.
//    2019); acc = lambda * eps.
//  * ev: an element-wise fp32 evaluation (a product, silu and its derivative, the rounding of
//    an fp64-exact value to fp32) lies within ev * |value|.
//  * gate: the fp32 softmax gate lies within gate * g.
struct FlipModel {
  double acc, ev, gate;
};

// Largest change of the bf16 rounding of v when v moves by at most dv.  Rounding is
// monotone, so the extremes are the roundings of v - dv and v + dv.
double round_spread(double v, double dv) {
  const double r = round_bf16(v);
  return std::fmax(std::fabs(round_bf16(v + dv) - r), std::fabs(round_bf16(v - dv) - r));
}

// Signed deviation interval of that rounding: round(v - dv) - round(v) <= 0 and
// round(v + dv) - round(v) >= 0.
struct Dev {
  double lo, hi;
  double mag() const { return std::fmax(-lo, hi); }
};
Dev round_dev(double v, double dv) {
  const double r = round_bf16(v);
  return Dev{round_bf16(v - dv) - r, round_bf16(v + dv) - r};
}

// Extremes of c * delta for delta in [lo, hi], added to an interval [dn, up].
inline void add_scaled(double c, const Dev& dv, double* dn, double* up) {
  const double p = c * dv.lo, q = c * dv.hi;
  *dn += std::fmin(p, q);
  *up += std::fmax(p, q);
}

// Lipschitz constants over the whole real line: |silu'(a)| <= 1.1, |silu''(a)| <= 0.5
// (the largest values are 1.0998 near a = 2.4 and 0.5 at a = 0).
constexpr double kSiluLip = 1.1;
constexpr double kSiluPrimeLip = 0.5;

// z = x y with x known to within dx and y to within dy: z is known to within
// |x| dy + |y| dx + dx dy.
inline double prod_unc(double x, double dx, double y, double dy) {
  return std::fabs(x) * dy + std::fabs(y) * dx + dx * dy;
}

// Flip intervals of h = bf16(silu(a) b) (bf16(relu(a)^2) without W3) of one pair, from its
// forward sums a, b [dff] and their trace: Dh [dff].
void h_flip_bounds(int dff, bool gated, const double* a, const double* b, const FwdTrace& ft,
                   const FlipModel& M, Dev* Dh) {
  for (int f = 0; f < dff; ++f) {
    const double dA = M.acc * std::sqrt(ft.sa[f]);
    const double dB = gated ? M.acc * std::sqrt(ft.sb[f]) : 0.0;
    const double s = gated ? a[f] * sigmoid(a[f]) : 0.0;  // silu(a)
    const double r = a[f] > 0.0 ? a[f] : 0.0;              // relu(a)
    const double dv = gated ? prod_unc(s, kSiluLip * dA, b[f], dB) : prod_unc(r, dA, r, dA);
    Dh[f] = round_dev(ft.vh[f], dv + M.ev * std::fabs(ft.vh[f]));
  }
}

// Flip intervals of the pair's bf16 output row o = bf16(h W2): Do [d].  The other
// implementation's pre-rounding o differs from the oracle's by its fp32 accumulation error and
// by every h flip times |W2| (its h is the oracle's up to those flips).
template <class V>
void o_flip_bounds(const V* W2e, int d, int dff, const FwdTrace& ft, const Dev* Dh,
                   const FlipModel& M, Dev* Do) {
  std::vector<double> dv(d);
  for (int c = 0; c < d; ++c) dv[c] = M.acc * std::sqrt(ft.so[c]);
  for (int f = 0; f < dff; ++f) {
    const double m = Dh[f].mag();
    if (m == 0.0) continue;
    const V* w2 = W2e + static_cast<int64_t>(f) * d;
    for (int c = 0; c < d; ++c) dv[c] += m * std::fabs(widen(w2[c]));
  }
  for (int c = 0; c < d; ++c) Do[c] = round_dev(ft.vo[c], dv[c]);
}

// Flip bounds of one token-expert pair: the signed intervals within which the other
// implementation's bf16 rounding of each operand lies around the oracle's.  In: the pair's
// gate g and dy [d]; the forward's a, b [dff] and their trace; the backward's dh [dff] and its
// trace.  Out: Dh [dff] (h), DdO [d] (dO = g dy), Dda [dff], Ddb [dff] (da, db; zero without
// W3).
template <class V>
void pair_flip_bounds(const V* W2e, int d, int dff, bool gated, double g, const double* dy,
                      const double* a, const double* b, const FwdTrace& ft, const double* dh,
                      const BwdTrace& bt, const FlipModel& M, Dev* Dh, Dev* DdO, Dev* Dda,
                      Dev* Ddb) {
  // dO: the fp32 product of the fp32 gate and dy, then bf16
  std::vector<int> flagged;  // columns c whose dO may round the other way
  for (int c = 0; c < d; ++c) {
    const double v = g * dy[c];
    DdO[c] = round_dev(v, std::fabs(dy[c]) * M.gate * g + M.ev * std::fabs(v));
    if (DdO[c].mag() != 0.0) flagged.push_back(c);
  }
  h_flip_bounds(dff, gated, a, b, ft, M, Dh);
  for (int f = 0; f < dff; ++f) {
    const double dA = M.acc * std::sqrt(ft.sa[f]);
    const double dB = gated ? M.acc * std::sqrt(ft.sb[f]) : 0.0;
    const double s = gated ? a[f] * sigmoid(a[f]) : 0.0;  // silu(a)
    const double r = a[f] > 0.0 ? a[f] : 0.0;              // relu(a)
    // dh = sum_c dO_c W2[f][c]: its accumulation error plus every dO flip times |W2|
    const V* w2 = W2e + static_cast<int64_t>(f) * d;
    double ddh = M.acc * std::sqrt(bt.sdh[f]);
    for (int c : flagged) ddh += DdO[c].mag() * std::fabs(widen(w2[c]));
    // da = dh q with q = b silu'(a) (2 relu(a) without W3); db = dh silu(a)
    double q, dq;
    if (gated) {
      const double sg = sigmoid(a[f]);
      const double sp = sg * (1.0 + a[f] * (1.0 - sg));
      q = b[f] * sp;
      dq = prod_unc(b[f], dB, sp, kSiluPrimeLip * dA);
    } else {
      q = 2.0 * r;
      dq = 2.0 * dA;
    }
    Dda[f] = round_dev(bt.vda[f], prod_unc(dh[f], ddh, q, dq) + M.ev * std::fabs(bt.vda[f]));
    Ddb[f] = gated ? round_dev(bt.vdb[f], prod_unc(dh[f], ddh, s, kSiluLip * dA) +
                                              M.ev * std::fabs(bt.vdb[f]))
                   : Dev{0.0, 0.0};
  }
}

struct Dims {
  int64_t T;
  int d, E, k, dff;
};

template <class V>
const V* w13(const V* W, const Dims& D, int e) {
  return W ? W + static_cast<int64_t>(e) * D.d * D.dff : nullptr;  // null: no W3
}
template <class V>
const V* w2of(const V* W, const Dims& D, int e) { return W + static_cast<int64_t>(e) * D.dff * D.d; }

bool dims_ok(int64_t T, int d, int E, int k, int dff) {
  return T >= 0 && d > 0 && E > 0 && k >= 1 && k <= E && dff > 0;
}

// Brute-force forward for a list of tokens: route each token, run its k experts on its own
// row, sum gate-weighted outputs.  With a flip model M (round_h on), also the rounding-flip
// allowance of each output element (ay [n,d]): the interval sum over j of g_j Do_jc, the flip
// interval of the pair's bf16 output row (which takes in the h flips), reported as
// max(up, -down).
template <class V>
int forward_tokens(const V* x, const double* logits, const V* W1, const V* W3, const V* W2,
                   const Dims& D, int round_h, const int64_t* tokens, int64_t n, double* y,
                   const FlipModel* M = nullptr, double* ay = nullptr) {
  if (M && !round_h) return -1;
  int bad = 0;
#pragma omp parallel
  {
    std::vector<int32_t> idx(D.k);
    std::vector<double> gate(D.k), a(D.dff), b(D.dff), h(D.dff), o(D.d);
    std::vector<double> sa, sb, vh, so, vo, ydn, yup;
    std::vector<Dev> Dh, Do;
    if (M) {
      for (auto* v : {&sa, &sb, &vh}) v->assign(D.dff, 0.0);
      for (auto* v : {&so, &vo, &ydn, &yup}) v->assign(D.d, 0.0);
      Dh.resize(D.dff);
      Do.resize(D.d);
    }
    const FwdTrace ft{sa.data(), sb.data(), vh.data(), so.data(), vo.data()};
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
      const int64_t t = tokens ? tokens[i] : i;
      if (t < 0 || t >= D.T) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      route_token(logits + t * D.E, D.E, D.k, idx.data(), gate.data());
      double* yt = y + i * D.d;
      for (int c = 0; c < D.d; ++c) yt[c] = 0.0;
      if (M) for (int c = 0; c < D.d; ++c) ydn[c] = yup[c] = 0.0;
      for (int j = 0; j < D.k; ++j) {
        const int e = idx[j];
        ffn_row(x + t * D.d, w13(W1, D, e), w13(W3, D, e), w2of(W2, D, e), D.d, D.dff, round_h,
                a.data(), b.data(), h.data(), o.data(), M ? &ft : nullptr);
        for (int c = 0; c < D.d; ++c) yt[c] += gate[j] * o[c];
        if (!M) continue;
        h_flip_bounds(D.dff, W3 != nullptr, a.data(), b.data(), ft, *M, Dh.data());
        o_flip_bounds(w2of(W2, D, e), D.d, D.dff, ft, Dh.data(), *M, Do.data());
        for (int c = 0; c < D.d; ++c) add_scaled(gate[j], Do[c], &ydn[c], &yup[c]);
      }
      if (M && ay)
        for (int c = 0; c < D.d; ++c) ay[i * D.d + c] = std::fmax(yup[c], -ydn[c]);
    }
  }
  return bad ? -1 : 0;
}

void route_all(const double* logits, const Dims& D, int32_t* idx, double* gate) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < D.T; ++t)
    route_token(logits + t * D.E, D.E, D.k, idx + t * D.k, gate + t * D.k);
}

// counts, exclusive offsets and the stable permutation (rows ordered by expert, then token).
void dispatch_all(const int32_t* idx, const Dims& D, int32_t* counts, int32_t* offsets,
                  int32_t* perm, int32_t* pos) {
  for (int e = 0; e < D.E; ++e) counts[e] = 0;
  for (int64_t p = 0; p < D.T * D.k; ++p) counts[idx[p]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < D.E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int64_t> fill(offsets, offsets + D.E);
  for (int64_t t = 0; t < D.T; ++t)
    for (int j = 0; j < D.k; ++j) {
      const int64_t p = t * D.k + j;
      const int64_t r = fill[idx[p]]++;
      perm[r] = static_cast<int32_t>(p);
      pos[p] = static_cast<int32_t>(r);
    }
}

// Permuted forward: route, dispatch, copy rows into expert order, run each row through its
// expert, combine back to token order.
template <class V>
int forward_permuted(const V* x, const double* logits, const V* W1, const V* W3, const V* W2,
                     const Dims& D, int round_h, double* y, V* x_perm_out, double* o_perm_out) {
  const int64_t P = D.T * D.k;
  std::vector<int32_t> idx(P), counts(D.E), offsets(D.E + 1), perm(P), pos(P);
  std::vector<double> gate(P);
  route_all(logits, D, idx.data(), gate.data());
  dispatch_all(idx.data(), D, counts.data(), offsets.data(), perm.data(), pos.data());
  std::vector<V> xp(static_cast<size_t>(P) * D.d);
  for (int64_t r = 0; r < P; ++r) {
    const int64_t t = perm[r] / D.k;
    for (int c = 0; c < D.d; ++c) xp[r * D.d + c] = x[t * D.d + c];
  }
  std::vector<int32_t> row_expert(P);
  for (int e = 0; e < D.E; ++e)
    for (int64_t r = offsets[e]; r < offsets[e + 1]; ++r) row_expert[r] = e;
  std::vector<double> op(static_cast<size_t>(P) * D.d);
#pragma omp parallel
  {
    std::vector<double> a(D.dff), b(D.dff), h(D.dff);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < P; ++r) {
      const int e = row_expert[r];
      ffn_row(xp.data() + r * D.d, w13(W1, D, e), w13(W3, D, e), w2of(W2, D, e), D.d, D.dff,
              round_h, a.data(), b.data(), h.data(), op.data() + r * D.d);
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < D.T; ++t) {
    double* yt = y + t * D.d;
    for (int c = 0; c < D.d; ++c) yt[c] = 0.0;
    for (int j = 0; j < D.k; ++j) {
      const double* orow = op.data() + static_cast<int64_t>(pos[t * D.k + j]) * D.d;
      const double g = gate[t * D.k + j];
      for (int c = 0; c < D.d; ++c) yt[c] += g * orow[c];
    }
  }
  if (x_perm_out) std::memcpy(x_perm_out, xp.data(), xp.size() * sizeof(V));
  if (o_perm_out) std::memcpy(o_perm_out, op.data(), op.size() * sizeof(double));
  return 0;
}

// Per-token backward (brute force): dx_t = sum_j dxp_j, dgate_t, and dlogits_t through the
// softmax over the selected logits: dl_{e_j} = g_j (dgate_j - sum_i g_i dgate_i), 0 elsewhere.
// With a flip model M (round_grad on), also the rounding-flip allowance of each output
// (adx [n,d], adg [n,k], adl [n,E]; null pointers skip one): the largest |change| of the
// output when every flagged operand takes any value of its deviation interval, namely
//   dx_t[c]:   sum_j sum_f W1[e_j][c][f] Dda_jf + W3[e_j][c][f] Ddb_jf,
//   dgate_tj:  sum_c dy_t[c] Do_jc (dgate reads the pair's bf16 output row o, whose flip
//              interval Do takes in the h flips),
//   dl_{e_j}:  sum_i c_ji dgate_ti, c_jj = g_j (1 - g_j), c_ji = -g_j g_i,
// each evaluated as an interval sum and reported as max(up, -down).
template <class V, class G>
int backward_tokens(const V* x, const double* logits, const V* W1, const V* W3, const V* W2,
                    const G* dy, const Dims& D, int round_h, int round_grad,
                    const int64_t* tokens, int64_t n, double* dx, double* dgate,
                    double* dlogits, const FlipModel* M = nullptr, double* adx = nullptr,
                    double* adg = nullptr, double* adl = nullptr) {
  if (M && !round_grad) return -1;
  int bad = 0;
#pragma omp parallel
  {
    std::vector<int32_t> idx(D.k);
    std::vector<double> gate(D.k), a(D.dff), b(D.dff), h(D.dff), o(D.d), dyv(D.d), dO(D.d),
        dh(D.dff), da(D.dff), db(D.dff), dxp(D.d);
    // flip-allowance work arrays
    std::vector<double> sa, sb, vh, so, vo, sdh, vda, vdb, xdn, xup, gdn, gup;
    std::vector<Dev> Dh, Do, DdO, Dda, Ddb;
    std::vector<int> live;
    if (M) {
      for (auto* v : {&sa, &sb, &vh, &sdh, &vda, &vdb}) v->assign(D.dff, 0.0);
      so.assign(D.d, 0.0);
      vo.assign(D.d, 0.0);
      Do.resize(D.d);
      Dh.resize(D.dff);
      Dda.resize(D.dff);
      Ddb.resize(D.dff);
      DdO.resize(D.d);
      xdn.assign(D.d, 0.0);
      xup.assign(D.d, 0.0);
      gdn.assign(D.k, 0.0);
      gup.assign(D.k, 0.0);
    }
    const FwdTrace ft{sa.data(), sb.data(), vh.data(), so.data(), vo.data()};
    const BwdTrace bt{sdh.data(), vda.data(), vdb.data()};
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
      const int64_t t = tokens ? tokens[i] : i;
      if (t < 0 || t >= D.T) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      route_token(logits + t * D.E, D.E, D.k, idx.data(), gate.data());
      for (int c = 0; c < D.d; ++c) dyv[c] = widen(dy[t * D.d + c]);
      double* dxt = dx ? dx + i * D.d : nullptr;
      if (dxt) for (int c = 0; c < D.d; ++c) dxt[c] = 0.0;
      if (M) {
        for (int c = 0; c < D.d; ++c) xdn[c] = xup[c] = 0.0;
      }
      std::vector<double> dg(D.k);
      for (int j = 0; j < D.k; ++j) {
        const int e = idx[j];
        ffn_row(x + t * D.d, w13(W1, D, e), w13(W3, D, e), w2of(W2, D, e), D.d, D.dff, round_h,
                a.data(), b.data(), h.data(), o.data(), M ? &ft : nullptr);
        ffn_row_bwd(w13(W1, D, e), w13(W3, D, e), w2of(W2, D, e), D.d, D.dff, gate[j],
                    dyv.data(), a.data(), b.data(), o.data(), round_grad, &dg[j], dO.data(),
                    dh.data(), da.data(), db.data(), dxp.data(), M ? &bt : nullptr);
        if (dxt) for (int c = 0; c < D.d; ++c) dxt[c] += dxp[c];
        if (!M) continue;
        const V* W1e = w13(W1, D, e);
        const V* W3e = w13(W3, D, e);
        const V* W2e = w2of(W2, D, e);
        pair_flip_bounds(W2e, D.d, D.dff, W3e != nullptr, gate[j], dyv.data(), a.data(),
                         b.data(), ft, dh.data(), bt, *M, Dh.data(), DdO.data(), Dda.data(),
                         Ddb.data());
        live.clear();  // columns f with a flagged da or db
        for (int f = 0; f < D.dff; ++f)
          if (Dda[f].mag() != 0.0 || Ddb[f].mag() != 0.0) live.push_back(f);
        for (int c = 0; c < D.d; ++c) {
          const V* w1 = W1e + static_cast<int64_t>(c) * D.dff;
          const V* w3 = W3e ? W3e + static_cast<int64_t>(c) * D.dff : nullptr;
          for (int f : live) {
            add_scaled(widen(w1[f]), Dda[f], &xdn[c], &xup[c]);
            if (w3) add_scaled(widen(w3[f]), Ddb[f], &xdn[c], &xup[c]);
          }
        }
        gdn[j] = gup[j] = 0.0;
        o_flip_bounds(W2e, D.d, D.dff, ft, Dh.data(), *M, Do.data());
        for (int c = 0; c < D.d; ++c) add_scaled(dyv[c], Do[c], &gdn[j], &gup[j]);
      }
      if (dgate) for (int j = 0; j < D.k; ++j) dgate[i * D.k + j] = dg[j];
      if (dlogits) {
        double* dl = dlogits + i * D.E;
        for (int e = 0; e < D.E; ++e) dl[e] = 0.0;
        double sgd = 0.0;
        for (int j = 0; j < D.k; ++j) sgd += gate[j] * dg[j];
        for (int j = 0; j < D.k; ++j) dl[idx[j]] = gate[j] * (dg[j] - sgd);
      }
      if (!M) continue;
      if (adx)
        for (int c = 0; c < D.d; ++c) adx[i * D.d + c] = std::fmax(xup[c], -xdn[c]);
      if (adg)
        for (int j = 0; j < D.k; ++j) adg[i * D.k + j] = std::fmax(gup[j], -gdn[j]);
      if (adl) {
        double* al = adl + i * D.E;
        for (int e = 0; e < D.E; ++e) al[e] = 0.0;
        for (int j = 0; j < D.k; ++j) {
          double dn = 0.0, up = 0.0;
          for (int q = 0; q < D.k; ++q) {
            const double cq = q == j ? gate[j] * (1.0 - gate[j]) : -gate[j] * gate[q];
            const Dev iv{gdn[q], gup[q]};
            add_scaled(cq, iv, &dn, &up);
          }
          al[idx[j]] = std::fmax(up, -dn);
        }
      }
    }
  }
  return bad ? -1 : 0;
}

// Weight gradients of selected experts, summed over every pair routed to them:
//   dW1[e] = sum x^T da, dW3[e] = sum x^T db, dW2[e] = sum h^T dO.
// With a flip model M (round_grad on), also their rounding-flip allowances (null skips one),
// interval sums over the expert's rows r:
//   dW1[c][f]: x_rc Dda_rf;  dW3[c][f]: x_rc Ddb_rf;
//   dW2[f][c]: (h_rf + dh) (dO_rc + ddO) - h_rf dO_rc over the corners of Dh_rf x DdO_rc.
template <class V, class G>
int backward_dw(const V* x, const double* logits, const V* W1, const V* W3, const V* W2,
                const G* dy, const Dims& D, int round_h, int round_grad, const int32_t* experts,
                int n_exp, double* dW1, double* dW3, double* dW2, const FlipModel* M = nullptr,
                double* a1 = nullptr, double* a3 = nullptr, double* a2 = nullptr) {
  if (M && !round_grad) return -1;
  const int64_t P = D.T * D.k;
  std::vector<int32_t> idx(P);
  std::vector<double> gate(P);
  route_all(logits, D, idx.data(), gate.data());
  for (int q = 0; q < n_exp; ++q) {
    const int e = experts[q];
    if (e < 0 || e >= D.E) return -1;
    std::vector<int64_t> pairs;  // pairs routed to e, in token order
    for (int64_t p = 0; p < P; ++p)
      if (idx[p] == e) pairs.push_back(p);
    const int64_t R = static_cast<int64_t>(pairs.size());
    std::vector<double> A(R * D.dff), B(R * D.dff), H(R * D.dff), DO(R * D.d), DA(R * D.dff),
        DB(R * D.dff);
    std::vector<Dev> fDh, fDdO, fDda, fDdb;  // per-row flip intervals
    if (M) {
      fDh.resize(R * D.dff);
      fDdO.resize(R * D.d);
      fDda.resize(R * D.dff);
      fDdb.resize(R * D.dff);
    }
#pragma omp parallel
    {
      std::vector<double> o(D.d), dyv(D.d), dh(D.dff), dxp(D.d);
      std::vector<double> sa, sb, vh, sdh, vda, vdb;
      if (M)
        for (auto* v : {&sa, &sb, &vh, &sdh, &vda, &vdb}) v->assign(D.dff, 0.0);
      const FwdTrace ft{sa.data(), sb.data(), vh.data()};
      const BwdTrace bt{sdh.data(), vda.data(), vdb.data()};
#pragma omp for schedule(dynamic, 1)
      for (int64_t r = 0; r < R; ++r) {
        const int64_t p = pairs[r], t = p / D.k;
        ffn_row(x + t * D.d, w13(W1, D, e), w13(W3, D, e), w2of(W2, D, e), D.d, D.dff, round_h,
                &A[r * D.dff], &B[r * D.dff], &H[r * D.dff], o.data(), M ? &ft : nullptr);
        for (int c = 0; c < D.d; ++c) dyv[c] = widen(dy[t * D.d + c]);
        double dg;
        ffn_row_bwd(w13(W1, D, e), w13(W3, D, e), w2of(W2, D, e), D.d, D.dff, gate[p], dyv.data(),
                    &A[r * D.dff], &B[r * D.dff], o.data(), round_grad, &dg, &DO[r * D.d],
                    dh.data(), &DA[r * D.dff], &DB[r * D.dff], dxp.data(), M ? &bt : nullptr);
        if (M)
          pair_flip_bounds(w2of(W2, D, e), D.d, D.dff, W3 != nullptr, gate[p], dyv.data(),
                           &A[r * D.dff], &B[r * D.dff], ft, dh.data(), bt, *M,
                           &fDh[r * D.dff], &fDdO[r * D.d], &fDda[r * D.dff], &fDdb[r * D.dff]);
      }
    }
    double* g1 = dW1 + static_cast<int64_t>(q) * D.d * D.dff;
    double* g3 = dW3 ? dW3 + static_cast<int64_t>(q) * D.d * D.dff : nullptr;  // null: no W3
    double* g2 = dW2 + static_cast<int64_t>(q) * D.dff * D.d;
    double* h1 = M && a1 ? a1 + static_cast<int64_t>(q) * D.d * D.dff : nullptr;
    double* h3 = M && a3 && W3 ? a3 + static_cast<int64_t>(q) * D.d * D.dff : nullptr;
    double* h2 = M && a2 ? a2 + static_cast<int64_t>(q) * D.dff * D.d : nullptr;
    // per row: the columns with a flagged da, db (f) and dO (c); only those add to an interval
    std::vector<std::vector<int>> nz_a(M ? R : 0), nz_b(M ? R : 0), nz_o(M ? R : 0);
    for (int64_t r = 0; M && r < R; ++r) {
      for (int f = 0; f < D.dff; ++f) {
        if (fDda[r * D.dff + f].mag() != 0.0) nz_a[r].push_back(f);
        if (fDdb[r * D.dff + f].mag() != 0.0) nz_b[r].push_back(f);
      }
      for (int c = 0; c < D.d; ++c)
        if (fDdO[r * D.d + c].mag() != 0.0) nz_o[r].push_back(c);
    }
#pragma omp parallel
    {
      std::vector<double> dn1, up1, dn3, up3;
      if (h1) { dn1.assign(D.dff, 0.0); up1.assign(D.dff, 0.0); }
      if (h3) { dn3.assign(D.dff, 0.0); up3.assign(D.dff, 0.0); }
#pragma omp for schedule(static)
      for (int c = 0; c < D.d; ++c) {
        double* r1 = g1 + static_cast<int64_t>(c) * D.dff;
        double* r3 = g3 ? g3 + static_cast<int64_t>(c) * D.dff : nullptr;
        for (int f = 0; f < D.dff; ++f) r1[f] = 0.0;
        if (r3) for (int f = 0; f < D.dff; ++f) r3[f] = 0.0;
        if (h1) for (int f = 0; f < D.dff; ++f) dn1[f] = up1[f] = 0.0;
        if (h3) for (int f = 0; f < D.dff; ++f) dn3[f] = up3[f] = 0.0;
        for (int64_t r = 0; r < R; ++r) {
          const double xc = widen(x[(pairs[r] / D.k) * D.d + c]);
          for (int f = 0; f < D.dff; ++f) r1[f] += xc * DA[r * D.dff + f];
          if (r3) for (int f = 0; f < D.dff; ++f) r3[f] += xc * DB[r * D.dff + f];
          if (h1)
            for (int f : nz_a[r]) add_scaled(xc, fDda[r * D.dff + f], &dn1[f], &up1[f]);
          if (h3)
            for (int f : nz_b[r]) add_scaled(xc, fDdb[r * D.dff + f], &dn3[f], &up3[f]);
        }
        if (h1)
          for (int f = 0; f < D.dff; ++f)
            h1[static_cast<int64_t>(c) * D.dff + f] = std::fmax(up1[f], -dn1[f]);
        if (h3)
          for (int f = 0; f < D.dff; ++f)
            h3[static_cast<int64_t>(c) * D.dff + f] = std::fmax(up3[f], -dn3[f]);
      }
    }
#pragma omp parallel
    {
      std::vector<double> dn2, up2;
      if (h2) { dn2.assign(D.d, 0.0); up2.assign(D.d, 0.0); }
#pragma omp for schedule(static)
      for (int f = 0; f < D.dff; ++f) {
        double* r2 = g2 + static_cast<int64_t>(f) * D.d;
        for (int c = 0; c < D.d; ++c) r2[c] = 0.0;
        if (h2) for (int c = 0; c < D.d; ++c) dn2[c] = up2[c] = 0.0;
        for (int64_t r = 0; r < R; ++r) {
          const double hf = H[r * D.dff + f];
          for (int c = 0; c < D.d; ++c) r2[c] += hf * DO[r * D.d + c];
          if (!h2) continue;
          const Dev dhf = fDh[r * D.dff + f];
          // (h + u)(dO + w) - h dO = u dO + h w + u w, extremes at the corners
          auto corners = [&](int c) {
            const Dev ddo = fDdO[r * D.d + c];
            const double dov = DO[r * D.d + c];
            double lo = 0.0, hi = 0.0;
            bool first = true;
            for (double u : {dhf.lo, dhf.hi})
              for (double w : {ddo.lo, ddo.hi}) {
                const double z = u * dov + hf * w + u * w;
                lo = first ? z : std::fmin(lo, z);
                hi = first ? z : std::fmax(hi, z);
                first = false;
              }
            dn2[c] += lo;
            up2[c] += hi;
          };
          if (dhf.mag() != 0.0) {
            for (int c = 0; c < D.d; ++c) corners(c);
          } else {
            for (int c : nz_o[r]) corners(c);  // only the dO flips of this row move dW2[f]
          }
        }
        if (h2)
          for (int c = 0; c < D.d; ++c)
            h2[static_cast<int64_t>(f) * D.d + c] = std::fmax(up2[c], -dn2[c]);
      }
    }
  }
  return 0;
}

// Operands of one token-expert pair (token t, slot j) and their flip intervals, for the tests
// of the allowance: h, its pre-rounding value vh and interval Dh [dff][2] (lo, hi); dO and
// DdO [d][2]; da, db and Dda, Ddb [dff][2]; the expert index and gate through e_out, g_out.
template <class V>
int pair_operands(const V* x, const double* logits, const V* W1, const V* W3, const V* W2,
                  const V* dy, const Dims& D, int64_t t, int j, const FlipModel& M, int* e_out,
                  double* g_out, double* h, double* vh, double* Dh, double* dO, double* DdO,
                  double* da, double* Dda, double* db, double* Ddb, double* o, double* Do) {
  if (t < 0 || t >= D.T || j < 0 || j >= D.k) return -1;
  std::vector<int32_t> idx(D.k);
  std::vector<double> gate(D.k), a(D.dff), b(D.dff), dyv(D.d), dh(D.dff), dxp(D.d),
      sa(D.dff), sb(D.dff), so(D.d), vo(D.d), sdh(D.dff), vda(D.dff), vdb(D.dff);
  std::vector<Dev> ih(D.dff), io(D.d), ia(D.dff), ib(D.dff), iy(D.d);
  route_token(logits + t * D.E, D.E, D.k, idx.data(), gate.data());
  const int e = idx[j];
  const FwdTrace ft{sa.data(), sb.data(), vh, so.data(), vo.data()};
  const BwdTrace bt{sdh.data(), vda.data(), vdb.data()};
  ffn_row(x + t * D.d, w13(W1, D, e), w13(W3, D, e), w2of(W2, D, e), D.d, D.dff, 1, a.data(),
          b.data(), h, o, &ft);
  for (int c = 0; c < D.d; ++c) dyv[c] = widen(dy[t * D.d + c]);
  double dg;
  ffn_row_bwd(w13(W1, D, e), w13(W3, D, e), w2of(W2, D, e), D.d, D.dff, gate[j], dyv.data(),
              a.data(), b.data(), o, 1, &dg, dO, dh.data(), da, db, dxp.data(), &bt);
  pair_flip_bounds(w2of(W2, D, e), D.d, D.dff, W3 != nullptr, gate[j], dyv.data(), a.data(),
                   b.data(), ft, dh.data(), bt, M, ih.data(), io.data(), ia.data(), ib.data());
  o_flip_bounds(w2of(W2, D, e), D.d, D.dff, ft, ih.data(), M, iy.data());
  for (int c = 0; c < D.d; ++c) {
    Do[2 * c] = iy[c].lo;
    Do[2 * c + 1] = iy[c].hi;
  }
  for (int f = 0; f < D.dff; ++f) {
    Dh[2 * f] = ih[f].lo;
    Dh[2 * f + 1] = ih[f].hi;
    Dda[2 * f] = ia[f].lo;
    Dda[2 * f + 1] = ia[f].hi;
    Ddb[2 * f] = ib[f].lo;
    Ddb[2 * f + 1] = ib[f].hi;
  }
  for (int c = 0; c < D.d; ++c) {
    DdO[2 * c] = io[c].lo;
    DdO[2 * c + 1] = io[c].hi;
  }
  *e_out = e;
  *g_out = gate[j];
  return 0;
}

// Flip-model accumulation bound of one plain sum: the running partial sums of t [n] (in index
// order) give acc * sqrt(sum_j s_j^2); the exact sum goes to *sum.
double sum_bound(const double* t, int64_t n, double acc, double* sum) {
  double s = 0.0, sq = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    s += t[i];
    sq += s * s;
  }
  *sum = s;
  return acc * std::sqrt(sq);
}

// ---------------------------------------------------------------------- FP8 dispatch
// Per-row E4M3 quantization of x [T][d] (bf16 bits): dequantized values q s into xq, the
// scales into s.
void quantize_rows(const uint16_t* x, int64_t T, int d, double* xq, double* s) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    double amax = 0.0;
    for (int c = 0; c < d; ++c) amax = std::fmax(amax, std::fabs(widen(x[t * d + c])));
    const double st = e4m3_scale(amax);
    s[t] = st;
    if (xq)
      for (int c = 0; c < d; ++c) xq[t * d + c] = e4m3_quant(widen(x[t * d + c]), st) * st;
  }
}

// Per-column E4M3 scales of W [E][K][N] (bf16 bits), over K: s [E][N].
void column_scales(const uint16_t* W, int E, int K, int N, double* s) {
#pragma omp parallel for schedule(static)
  for (int64_t en = 0; en < static_cast<int64_t>(E) * N; ++en) {
    const int64_t e = en / N, n = en % N;
    double amax = 0.0;
    for (int c = 0; c < K; ++c)
      amax = std::fmax(amax, std::fabs(widen(W[(e * K + c) * N + n])));
    s[en] = e4m3_scale(amax);
  }
}

// Forward with the FP8 dispatch payload: each token's row and the first projections' weights
// quantized as above (weights quantized where they are used), SwiGLU, bf16 h, bf16 W2, and
// (round_h) the bf16 output row, as in ffn_row.  With a flip model M (round_h on), also the
// rounding-flip allowance of each output element (ay [n,d]), as in forward_tokens: a and b
// are the sums of the dequantized products, traced like ffn_row's.
int forward_tokens_fp8(const uint16_t* x, const double* logits, const uint16_t* W1,
                       const uint16_t* W3, const uint16_t* W2, const Dims& D, int round_h,
                       const int64_t* tokens, int64_t n, double* y,
                       const FlipModel* M = nullptr, double* ay = nullptr) {
  if (M && !round_h) return -1;
  std::vector<double> s1(static_cast<size_t>(D.E) * D.dff), s3(s1.size());
  column_scales(W1, D.E, D.d, D.dff, s1.data());
  column_scales(W3, D.E, D.d, D.dff, s3.data());
  int bad = 0;
#pragma omp parallel
  {
    std::vector<int32_t> idx(D.k);
    std::vector<double> gate(D.k), xq(D.d), a(D.dff), b(D.dff), h(D.dff), o(D.d);
    std::vector<double> sa(D.dff), sb(D.dff), vh(D.dff), so(D.d), vo(D.d), ydn(D.d), yup(D.d);
    std::vector<Dev> Dh(D.dff), Do(D.d);
    const FwdTrace ft{sa.data(), sb.data(), vh.data(), so.data(), vo.data()};
    double st;
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
      const int64_t t = tokens ? tokens[i] : i;
      if (t < 0 || t >= D.T) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      quantize_rows(x + t * D.d, 1, D.d, xq.data(), &st);
      route_token(logits + t * D.E, D.E, D.k, idx.data(), gate.data());
      double* yt = y + i * D.d;
      for (int c = 0; c < D.d; ++c) yt[c] = ydn[c] = yup[c] = 0.0;
      for (int j = 0; j < D.k; ++j) {
        const int e = idx[j];
        const uint16_t* w1 = w13(W1, D, e);
        const uint16_t* w3 = w13(W3, D, e);
        const double* s1e = s1.data() + static_cast<int64_t>(e) * D.dff;
        const double* s3e = s3.data() + static_cast<int64_t>(e) * D.dff;
        for (int f = 0; f < D.dff; ++f) { a[f] = 0.0; b[f] = 0.0; sa[f] = 0.0; sb[f] = 0.0; }
        for (int c = 0; c < D.d; ++c) {
          const uint16_t* r1 = w1 + static_cast<int64_t>(c) * D.dff;
          const uint16_t* r3 = w3 + static_cast<int64_t>(c) * D.dff;
          for (int f = 0; f < D.dff; ++f) {
            a[f] += xq[c] * (e4m3_quant(widen(r1[f]), s1e[f]) * s1e[f]);
            b[f] += xq[c] * (e4m3_quant(widen(r3[f]), s3e[f]) * s3e[f]);
          }
          if (M)
            for (int f = 0; f < D.dff; ++f) {
              sa[f] += a[f] * a[f];
              sb[f] += b[f] * b[f];
            }
        }
        for (int f = 0; f < D.dff; ++f) {
          const double hv = a[f] / (1.0 + std::exp(-a[f])) * b[f];
          vh[f] = hv;
          h[f] = round_h ? round_bf16(hv) : hv;
        }
        const uint16_t* w2 = w2of(W2, D, e);
        for (int c = 0; c < D.d; ++c) o[c] = so[c] = 0.0;
        for (int f = 0; f < D.dff; ++f) {
          for (int c = 0; c < D.d; ++c) o[c] += h[f] * widen(w2[static_cast<int64_t>(f) * D.d + c]);
          if (M) for (int c = 0; c < D.d; ++c) so[c] += o[c] * o[c];
        }
        for (int c = 0; c < D.d; ++c) {
          vo[c] = o[c];
          yt[c] += gate[j] * (round_h ? round_bf16(o[c]) : o[c]);
        }
        if (!M) continue;
        h_flip_bounds(D.dff, true, a.data(), b.data(), ft, *M, Dh.data());
        o_flip_bounds(w2, D.d, D.dff, ft, Dh.data(), *M, Do.data());
        for (int c = 0; c < D.d; ++c) add_scaled(gate[j], Do[c], &ydn[c], &yup[c]);
      }
      if (M && ay)
        for (int c = 0; c < D.d; ++c) ay[i * D.d + c] = std::fmax(yup[c], -ydn[c]);
    }
  }
  return bad ? -1 : 0;
}

}  // namespace

extern "C" {

int oracle_num_threads(void) { return omp_get_max_threads(); }

double oracle_round_bf16(double v) { return round_bf16(v); }

double oracle_round_e4m3(double v) { return round_e4m3(v); }

// Row quantization of x [T][d] (bf16 bits): dequantized values (or NULL) and row scales.
int oracle_quantize_rows_e4m3(const uint16_t* x, int64_t T, int d, double* xq, double* s) {
  if (T < 0 || d <= 0) return -1;
  quantize_rows(x, T, d, xq, s);
  return 0;
}

// Column quantization of W [E][K][N] (bf16 bits): E4M3 values (not dequantized) and the
// per-(expert, column) scales.
int oracle_quantize_cols_e4m3(const uint16_t* W, int E, int K, int N, double* q, double* s) {
  if (E <= 0 || K <= 0 || N <= 0) return -1;
  column_scales(W, E, K, N, s);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < static_cast<int64_t>(E) * K * N; ++i) {
    const int64_t e = i / (static_cast<int64_t>(K) * N), n = i % N;
    q[i] = e4m3_quant(widen(W[i]), s[e * N + n]);
  }
  return 0;
}

int oracle_route(const double* logits, int64_t T, int E, int k, int32_t* idx, double* gate) {
  if (!dims_ok(T, 1, E, k, 1)) return -1;
  Dims D{T, 1, E, k, 1};
  route_all(logits, D, idx, gate);
  return 0;
}

int oracle_dispatch(const int32_t* idx, int64_t T, int E, int k, int32_t* counts,
                    int32_t* offsets, int32_t* perm, int32_t* pos) {
  if (!dims_ok(T, 1, E, k, 1)) return -1;
  for (int64_t p = 0; p < T * k; ++p)
    if (idx[p] < 0 || idx[p] >= E) return -1;
  Dims D{T, 1, E, k, 1};
  dispatch_all(idx, D, counts, offsets, perm, pos);
  return 0;
}

#define ORACLE_DIMS int64_t T, int d, int E, int k, int dff

int oracle_forward_tokens_bf16(const uint16_t* x, const double* logits, const uint16_t* W1,
                               const uint16_t* W3, const uint16_t* W2, ORACLE_DIMS, int round_h,
                               const int64_t* tokens, int64_t n, double* y) {
  if (!dims_ok(T, d, E, k, dff)) return -1;
  return forward_tokens(x, logits, W1, W3, W2, Dims{T, d, E, k, dff}, round_h, tokens, n, y);
}

int oracle_forward_tokens_f64(const double* x, const double* logits, const double* W1,
                              const double* W3, const double* W2, ORACLE_DIMS, int round_h,
                              const int64_t* tokens, int64_t n, double* y) {
  if (!dims_ok(T, d, E, k, dff)) return -1;
  return forward_tokens(x, logits, W1, W3, W2, Dims{T, d, E, k, dff}, round_h, tokens, n, y);
}

int oracle_forward_permuted_bf16(const uint16_t* x, const double* logits, const uint16_t* W1,
                                 const uint16_t* W3, const uint16_t* W2, ORACLE_DIMS, int round_h,
                                 double* y, uint16_t* x_perm, double* o_perm) {
  if (!dims_ok(T, d, E, k, dff)) return -1;
  return forward_permuted(x, logits, W1, W3, W2, Dims{T, d, E, k, dff}, round_h, y, x_perm,
                          o_perm);
}

int oracle_backward_tokens_bf16(const uint16_t* x, const double* logits, const uint16_t* W1,
                                const uint16_t* W3, const uint16_t* W2, const uint16_t* dy,
                                ORACLE_DIMS, int round_h, int round_grad,
                                const int64_t* tokens, int64_t n, double* dx, double* dgate,
                                double* dlogits) {
  if (!dims_ok(T, d, E, k, dff)) return -1;
  return backward_tokens(x, logits, W1, W3, W2, dy, Dims{T, d, E, k, dff}, round_h, round_grad,
                         tokens, n, dx, dgate, dlogits);
}

int oracle_backward_tokens_f64(const double* x, const double* logits, const double* W1,
                               const double* W3, const double* W2, const double* dy, ORACLE_DIMS,
                               int round_h, int round_grad, const int64_t* tokens, int64_t n,
                               double* dx, double* dgate, double* dlogits) {
  if (!dims_ok(T, d, E, k, dff)) return -1;
  return backward_tokens(x, logits, W1, W3, W2, dy, Dims{T, d, E, k, dff}, round_h, round_grad,
                         tokens, n, dx, dgate, dlogits);
}

int oracle_backward_dw_bf16(const uint16_t* x, const double* logits, const uint16_t* W1,
                            const uint16_t* W3, const uint16_t* W2, const uint16_t* dy,
                            ORACLE_DIMS, int round_h, int round_grad, const int32_t* experts,
                            int n_exp, double* dW1, double* dW3, double* dW2) {
  if (!dims_ok(T, d, E, k, dff)) return -1;
  return backward_dw(x, logits, W1, W3, W2, dy, Dims{T, d, E, k, dff}, round_h, round_grad,
                     experts, n_exp, dW1, dW3, dW2);
}

int oracle_backward_dw_f64(const double* x, const double* logits, const double* W1,
                           const double* W3, const double* W2, const double* dy, ORACLE_DIMS,
                           int round_h, int round_grad, const int32_t* experts, int n_exp,
                           double* dW1, double* dW3, double* dW2) {
  if (!dims_ok(T, d, E, k, dff)) return -1;
  return backward_dw(x, logits, W1, W3, W2, dy, Dims{T, d, E, k, dff}, round_h, round_grad,
                     experts, n_exp, dW1, dW3, dW2);
}

// ------------------------------------------------ rounding-flip allowance (test bound)
// model = {acc, ev, gate} (FlipModel); round_grad is on.

double oracle_round_spread_bf16(double v, double dv) { return round_spread(v, dv); }

double oracle_sum_bound(const double* t, int64_t n, double acc, double* sum) {
  return sum_bound(t, n, acc, sum);
}

int oracle_forward_tokens_flip_bf16(const uint16_t* x, const double* logits, const uint16_t* W1,
                                    const uint16_t* W3, const uint16_t* W2, ORACLE_DIMS,
                                    const double* model, const int64_t* tokens, int64_t n,
                                    double* y, double* ay) {
  if (!dims_ok(T, d, E, k, dff) || !model) return -1;
  const FlipModel M{model[0], model[1], model[2]};
  return forward_tokens(x, logits, W1, W3, W2, Dims{T, d, E, k, dff}, 1, tokens, n, y, &M, ay);
}

int oracle_backward_tokens_flip_bf16(const uint16_t* x, const double* logits,
                                     const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                                     const uint16_t* dy, ORACLE_DIMS, int round_h,
                                     const double* model, const int64_t* tokens, int64_t n,
                                     double* dx, double* dgate, double* dlogits, double* adx,
                                     double* adg, double* adl) {
  if (!dims_ok(T, d, E, k, dff) || !model) return -1;
  const FlipModel M{model[0], model[1], model[2]};
  return backward_tokens(x, logits, W1, W3, W2, dy, Dims{T, d, E, k, dff}, round_h, 1, tokens,
                         n, dx, dgate, dlogits, &M, adx, adg, adl);
}

int oracle_backward_dw_flip_bf16(const uint16_t* x, const double* logits, const uint16_t* W1,
                                 const uint16_t* W3, const uint16_t* W2, const uint16_t* dy,
                                 ORACLE_DIMS, int round_h, const double* model,
                                 const int32_t* experts, int n_exp, double* dW1, double* dW3,
                                 double* dW2, double* a1, double* a3, double* a2) {
  if (!dims_ok(T, d, E, k, dff) || !model) return -1;
  const FlipModel M{model[0], model[1], model[2]};
  return backward_dw(x, logits, W1, W3, W2, dy, Dims{T, d, E, k, dff}, round_h, 1, experts,
                     n_exp, dW1, dW3, dW2, &M, a1, a3, a2);
}

int oracle_pair_operands_bf16(const uint16_t* x, const double* logits, const uint16_t* W1,
                              const uint16_t* W3, const uint16_t* W2, const uint16_t* dy,
                              ORACLE_DIMS, int64_t t, int j, const double* model, int* e_out,
                              double* g_out, double* h, double* vh, double* Dh, double* dO,
                              double* DdO, double* da, double* Dda, double* db, double* Ddb,
                              double* o, double* Do) {
  if (!dims_ok(T, d, E, k, dff) || !model) return -1;
  const FlipModel M{model[0], model[1], model[2]};
  return pair_operands(x, logits, W1, W3, W2, dy, Dims{T, d, E, k, dff}, t, j, M, e_out, g_out,
                       h, vh, Dh, dO, DdO, da, Dda, db, Ddb, o, Do);
}

int oracle_forward_tokens_fp8(const uint16_t* x, const double* logits, const uint16_t* W1,
                              const uint16_t* W3, const uint16_t* W2, ORACLE_DIMS, int round_h,
                              const int64_t* tokens, int64_t n, double* y) {
  if (!dims_ok(T, d, E, k, dff) || !W3) return -1;
  return forward_tokens_fp8(x, logits, W1, W3, W2, Dims{T, d, E, k, dff}, round_h, tokens, n, y);
}

// forward_tokens_fp8 (h and the output rows rounded) with its rounding-flip allowance ay [n,d]
int oracle_forward_tokens_fp8_flip(const uint16_t* x, const double* logits, const uint16_t* W1,
                                   const uint16_t* W3, const uint16_t* W2, ORACLE_DIMS,
                                   const double* model, const int64_t* tokens, int64_t n,
                                   double* y, double* ay) {
  if (!dims_ok(T, d, E, k, dff) || !W3 || !model) return -1;
  const FlipModel M{model[0], model[1], model[2]};
  return forward_tokens_fp8(x, logits, W1, W3, W2, Dims{T, d, E, k, dff}, 1, tokens, n, y, &M,
                            ay);
}

}  // extern "C"

// oracle.cpp — plain fp64 CPU primitives for the parallel transformer block oracle.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this
// library: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg do.
// It shares no code, header, table or helper with the CUDA path.
//
// The method (MegaScale: Scaling Large Language Model Training to More Than 10,000 GPUs,
// reading notes, section 1.1 "Parallel Transformer Block", eq. (4)) is
//     y = x + MLP(LN(x)) + Attention(LN(x)),
// with the MLP of the Megatron-LM tensor-parallel notes (section 2.1: Y = GeLU(XA)B,
// A:[h,4h], B:[4h,h]) and sliding-window attention (section 1.1 "Sliding Window
// Attention", eqs. (5)-(6): each token attends to the most recent w tokens).
//
// Every routine here computes its textbook definition directly, in double precision,
// with no rounding to bf16 anywhere. The block itself is composed step by step, in the
// pages' order, by oracle/oracle.py.
//
// Threads: rows are split into contiguous ranges, one per std::thread. Splitting rows
// changes no arithmetic: every output element is computed by one thread, summing its
// terms in ascending index order.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

int resolve_threads(int requested) {
  if (requested > 0) return requested;
  unsigned hc = std::thread::hardware_concurrency();
  return hc == 0 ? 1 : (int)hc;
}

// Calls body(begin, end) on `threads` contiguous slices of [0, n).
template <class Body>
void for_row_ranges(int64_t n, int threads, Body body) {
  threads = resolve_threads(threads);
  if (n <= 0) return;
  if (threads > n) threads = (int)n;
  if (threads == 1) {
    body((int64_t)0, n);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(threads);
  for (int t = 0; t < threads; ++t) {
    int64_t b = n * t / threads, e = n * (t + 1) / threads;
    pool.emplace_back([=] { body(b, e); });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Number of worker threads a call with `requested` (<= 0: all hardware threads) uses.
int oracle_threads(int requested) { return resolve_threads(requested); }

// LayerNorm over the last dimension (the "LN" of eq. (4)):
//   mu = mean_c x[r,c];  var = mean_c (x[r,c] - mu)^2   (biased, divide by H)
//   out[r,c] = (x[r,c] - mu) / sqrt(var + eps) * gamma[c] + beta[c]
void oracle_layernorm(int64_t rows, int64_t H, const double* x, const double* gamma,
                      const double* beta, double eps, double* out, int threads) {
  for_row_ranges(rows, threads, [=](int64_t r0, int64_t r1) {
    for (int64_t r = r0; r < r1; ++r) {
      const double* xr = x + r * H;
      double sum = 0.0;
      for (int64_t c = 0; c < H; ++c) sum += xr[c];
      const double mu = sum / (double)H;
      double sq = 0.0;
      for (int64_t c = 0; c < H; ++c) sq += (xr[c] - mu) * (xr[c] - mu);
      const double var = sq / (double)H;
      const double inv = 1.0 / std::sqrt(var + eps);
      double* o = out + r * H;
      for (int64_t c = 0; c < H; ++c) o[c] = (xr[c] - mu) * inv * gamma[c] + beta[c];
    }
  });
}

// RMSNorm over the last dimension (the normalisation of the fused "RMSNorm" kernel the
// MegaScale reading notes list in section 1.3; the pages do not define it, this is the
// standard form): out[r,c] = x[r,c] / sqrt(mean_c x[r,c]^2 + eps) * gamma[c].
void oracle_rmsnorm(int64_t rows, int64_t H, const double* x, const double* gamma, double eps,
                    double* out, int threads) {
  for_row_ranges(rows, threads, [=](int64_t r0, int64_t r1) {
    for (int64_t r = r0; r < r1; ++r) {
      const double* xr = x + r * H;
      double sq = 0.0;
      for (int64_t c = 0; c < H; ++c) sq += xr[c] * xr[c];
      const double inv = 1.0 / std::sqrt(sq / (double)H + eps);
      double* o = out + r * H;
      for (int64_t c = 0; c < H; ++c) o[c] = xr[c] * inv * gamma[c];
    }
  });
}

// Linear layer in the pages' convention Y = X W (Megatron-LM notes section 2.1, with W
// stored [in, out] row-major):
//   C[i, j] = bias[j] + sum_{k=0}^{K-1} A[i, k] * W[k, j]      (bias may be NULL)
// A is [M, K] with row stride lda, W is [K, N] with row stride ldw, C is [M, N] with
// row stride ldc. Rows are visited 16 at a time and columns 512 at a time so that each
// weight element fetched from memory serves 16 rows; within that, every C[i, j] still
// adds its K products in ascending k, starting from the bias (or 0).
void oracle_linear(int64_t M, int64_t K, int64_t N, const double* A, int64_t lda,
                   const double* W, int64_t ldw, const double* bias, double* C, int64_t ldc,
                   int threads) {
  const int64_t RB = 16, CB = 512;
  const int64_t n_groups = (M + RB - 1) / RB;
  for_row_ranges(n_groups, threads, [=](int64_t g0, int64_t g1) {
    for (int64_t g = g0; g < g1; ++g) {
      const int64_t i0 = g * RB, i1 = std::min(M, i0 + RB);
      for (int64_t j0 = 0; j0 < N; j0 += CB) {
        const int64_t j1 = std::min(N, j0 + CB);
        for (int64_t i = i0; i < i1; ++i)
          for (int64_t j = j0; j < j1; ++j) C[i * ldc + j] = bias ? bias[j] : 0.0;
        for (int64_t k = 0; k < K; ++k) {
          const double* wk = W + k * ldw;
          for (int64_t i = i0; i < i1; ++i) {
            const double a = A[i * lda + k];
            double* ci = C + i * ldc;
            for (int64_t j = j0; j < j1; ++j) ci[j] += a * wk[j];
          }
        }
      }
    }
  });
}

// Exact GeLU (the activation of Y = GeLU(XA)B): gelu(z) = z * Phi(z) = 0.5 z (1 + erf(z/sqrt 2)).
void oracle_gelu(int64_t n, const double* in, double* out, int threads) {
  const double inv_sqrt2 = 0.70710678118654752440;
  for_row_ranges(n, threads, [=](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i) out[i] = 0.5 * in[i] * (1.0 + std::erf(in[i] * inv_sqrt2));
  });
}

// SwiGLU activation (the "SiLU + elementwise multiply" fusion of section 1.3):
// out[i] = silu(gate[i]) * up[i],  silu(z) = z / (1 + exp(-z)).
void oracle_swiglu(int64_t n, const double* gate, const double* up, double* out, int threads) {
  for_row_ranges(n, threads, [=](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i) out[i] = gate[i] / (1.0 + std::exp(-gate[i])) * up[i];
  });
}

// FP8 E4M3 (the "E4M3" format of the performance notes, "BF16 / FP16 / FP8": 1 sign bit,
// 4 exponent bits with bias 7, 3 mantissa bits; no infinities; largest finite 448 =
// 1.75 * 2^8; smallest normal 2^-6; subnormals m * 2^-9, m = 1..7). Rounds v to the
// nearest representable value, ties to the even mantissa, and saturates at +-448.
// Returns the 8-bit code; *value gets the decoded value.
static uint8_t e4m3_round(double v, double* value) {
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(v);
  if (std::isnan(v)) a = 0.0;  // never produced by the callers below
  uint8_t code;
  double q;
  if (a < std::ldexp(1.0, -6)) {
    // subnormal grid, step 2^-9 (m = 8 reaches the smallest normal, code 0x08)
    const double m = std::nearbyint(a * 512.0);  // round half to even (default mode)
    q = m / 512.0;
    code = uint8_t(m);  // m in 0..8; 8 encodes exponent 1, mantissa 0
  } else {
    int e;
    std::frexp(a, &e);   // a = f * 2^e, f in [0.5, 1)
    const int ex = e - 1;  // a in [2^ex, 2^(ex+1))
    const double step = std::ldexp(1.0, ex - 3);
    q = std::nearbyint(a / step) * step;  // may reach 2^(ex+1): still representable
    if (q > 448.0) q = 448.0;
    int qe;
    const double qf = std::frexp(q, &qe);  // q = qf * 2^qe
    const int E = qe - 1;                  // q in [2^E, 2^(E+1))
    const int mant = int(std::nearbyint((qf * 2.0 - 1.0) * 8.0));
    code = uint8_t(((E + 7) << 3) | mant);
  }
  *value = sign ? -q : q;
  return uint8_t(sign | code);
}

// Per-row current scaling to E4M3, the same fp32 steps as the GPU quantizer:
//   amax = max_c |float(x[r,c])|,  inv = 448.0f / amax,  s[r] = amax / 448.0f   (fp32)
//   code[r,c] = e4m3(float(x[r,c]) * inv),  deq[r,c] = e4m3 value * s[r]
// (amax = 0: inv = s = 0, codes 0). deq may be NULL.
void oracle_quantize_e4m3_rows(int64_t rows, int64_t cols, const double* x, uint8_t* codes,
                               float* scales, double* deq, int threads) {
  for_row_ranges(rows, threads, [=](int64_t r0, int64_t r1) {
    for (int64_t r = r0; r < r1; ++r) {
      const double* xr = x + r * cols;
      float amax = 0.0f;
      for (int64_t c = 0; c < cols; ++c) amax = std::max(amax, std::fabs(float(xr[c])));
      const float inv = amax > 0.0f ? 448.0f / amax : 0.0f;
      const float s = amax / 448.0f;
      scales[r] = s;
      for (int64_t c = 0; c < cols; ++c) {
        const float t = float(xr[c]) * inv;
        double q;
        codes[r * cols + c] = e4m3_round(double(t), &q);
        if (deq) deq[r * cols + c] = q * double(s);
      }
    }
  });
}

// Sliding-window causal multi-head attention for ONE sequence (eqs. (5)-(6): each token
// attends only to the most recent w tokens, itself included).
//
// Queries: nq rows at sequence positions q_pos[]; keys/values: nk rows at positions
// k_pos[]. q, k, v and out are row-major with row length nh*dh; head j owns columns
// [j*dh, (j+1)*dh). Key kk is visible to query qq iff 0 <= q_pos[qq] - k_pos[kk] < w.
// For every query row and head:
//   s_kk = (q . k_kk) / sqrt(dh) for visible keys, -inf otherwise
//   p    = exp(s - max s) / sum exp(s - max s)                 (explicit softmax)
//   out  = sum_kk p_kk v_kk
// A query with no visible key (impossible when its own position is among k_pos) gets 0.
void oracle_swa_attention(int64_t nq, const int64_t* q_pos, const double* q, int64_t nk,
                          const int64_t* k_pos, const double* k, const double* v, int64_t nh,
                          int64_t dh, int64_t w, double* out, int threads) {
  const int64_t H = nh * dh;
  const double scale = 1.0 / std::sqrt((double)dh);
  const double neg_inf = -std::numeric_limits<double>::infinity();
  for_row_ranges(nq, threads, [=](int64_t r0, int64_t r1) {
    std::vector<double> s(nk > 0 ? nk : 1);
    for (int64_t qi = r0; qi < r1; ++qi) {
      for (int64_t head = 0; head < nh; ++head) {
        const double* qr = q + qi * H + head * dh;
        double smax = neg_inf;
        for (int64_t kk = 0; kk < nk; ++kk) {
          const int64_t dist = q_pos[qi] - k_pos[kk];
          if (dist < 0 || dist >= w) {
            s[kk] = neg_inf;
            continue;
          }
          const double* kr = k + kk * H + head * dh;
          double dot = 0.0;
          for (int64_t d = 0; d < dh; ++d) dot += qr[d] * kr[d];
          s[kk] = dot * scale;
          smax = std::max(smax, s[kk]);
        }
        double* o = out + qi * H + head * dh;
        for (int64_t d = 0; d < dh; ++d) o[d] = 0.0;
        if (smax == neg_inf) continue;
        double denom = 0.0;
        for (int64_t kk = 0; kk < nk; ++kk) {
          s[kk] = (s[kk] == neg_inf) ? 0.0 : std::exp(s[kk] - smax);
          denom += s[kk];
        }
        for (int64_t kk = 0; kk < nk; ++kk) {
          if (s[kk] == 0.0) continue;
          const double p = s[kk] / denom;
          const double* vr = v + kk * H + head * dh;
          for (int64_t d = 0; d < dh; ++d) o[d] += p * vr[d];
        }
      }
    }
  });
}

// ---------------------------------------------------------------------------- backward
// The backward pass of the block (training: MFU counts the forward's 2 and the backward's
// 4 FLOPs per weight and token, performance notes "MFU"). Each routine is the derivative
// of the forward routine above, written from the chain rule.

// LayerNorm / RMSNorm backward. With xhat = (x - mu) * rstd (RMSNorm: mu = 0,
// rstd = 1 / sqrt(mean x^2 + eps)) and g = dout * gamma:
//   dx[r,c] = rstd * (g[c] - mean_c g - xhat[c] * mean_c(g * xhat))   (RMSNorm: no mean_c g)
//   dgamma[c] = sum_r dout[r,c] * xhat[r,c],   dbeta[c] = sum_r dout[r,c]
// Rows are split over threads for dx; dgamma and dbeta are then summed per column, rows
// in ascending order. dbeta may be NULL.
void oracle_norm_backward(int64_t rows, int64_t H, const double* x, const double* gamma,
                          const double* dout, double eps, int rms, double* dx, double* dgamma,
                          double* dbeta, int threads) {
  std::vector<double> mu(rows > 0 ? rows : 1), rstd(rows > 0 ? rows : 1);
  for_row_ranges(rows, threads, [&](int64_t r0, int64_t r1) {
    std::vector<double> xhat(H), g(H);
    for (int64_t r = r0; r < r1; ++r) {
      const double* xr = x + r * H;
      double m = 0.0;
      if (!rms) {
        for (int64_t c = 0; c < H; ++c) m += xr[c];
        m /= (double)H;
      }
      double sq = 0.0;
      for (int64_t c = 0; c < H; ++c) sq += (xr[c] - m) * (xr[c] - m);
      const double rs = 1.0 / std::sqrt(sq / (double)H + eps);
      mu[r] = m;
      rstd[r] = rs;
      double mean_g = 0.0, mean_gx = 0.0;
      for (int64_t c = 0; c < H; ++c) {
        xhat[c] = (xr[c] - m) * rs;
        g[c] = dout[r * H + c] * gamma[c];
        mean_g += g[c];
        mean_gx += g[c] * xhat[c];
      }
      mean_g /= (double)H;
      mean_gx /= (double)H;
      if (rms) mean_g = 0.0;
      for (int64_t c = 0; c < H; ++c) dx[r * H + c] = rs * (g[c] - mean_g - xhat[c] * mean_gx);
    }
  });
  for_row_ranges(H, threads, [&](int64_t c0, int64_t c1) {
    for (int64_t c = c0; c < c1; ++c) {
      double sg = 0.0, sb = 0.0;
      for (int64_t r = 0; r < rows; ++r) {
        const double d = dout[r * H + c];
        sg += d * (x[r * H + c] - mu[r]) * rstd[r];
        sb += d;
      }
      dgamma[c] = sg;
      if (dbeta) dbeta[c] = sb;
    }
  });
}

// Exact GeLU backward: gelu'(z) = Phi(z) + z * phi(z), phi(z) = exp(-z^2 / 2) / sqrt(2 pi);
// dz[i] = dout[i] * gelu'(z[i]).
void oracle_gelu_backward(int64_t n, const double* z, const double* dout, double* dz,
                          int threads) {
  const double inv_sqrt2 = 0.70710678118654752440, inv_sqrt_2pi = 0.39894228040143267794;
  for_row_ranges(n, threads, [=](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i) {
      const double Phi = 0.5 * (1.0 + std::erf(z[i] * inv_sqrt2));
      const double phi = std::exp(-0.5 * z[i] * z[i]) * inv_sqrt_2pi;
      dz[i] = dout[i] * (Phi + z[i] * phi);
    }
  });
}

// SwiGLU backward for out = silu(gate) * up, silu(z) = z * sigma(z):
//   dup = dout * silu(gate),   dgate = dout * up * sigma(gate) * (1 + gate * (1 - sigma(gate)))
void oracle_swiglu_backward(int64_t n, const double* gate, const double* up, const double* dout,
                            double* dgate, double* dup, int threads) {
  for_row_ranges(n, threads, [=](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i) {
      const double sg = 1.0 / (1.0 + std::exp(-gate[i]));
      dup[i] = dout[i] * gate[i] * sg;
      dgate[i] = dout[i] * up[i] * sg * (1.0 + gate[i] * (1.0 - sg));
    }
  });
}

// Backward of oracle_swa_attention over ONE whole sequence of S tokens (positions 0..S-1),
// from its definition. Per head and query i, with the visible keys W(i) = {j : 0 <= i - j
// < w}, s_j = q_i . k_j / sqrt(dh), p = softmax(s) over W(i), o_i = sum_j p_j v_j:
//   dv_j += p_j do_i
//   dp_j  = do_i . v_j
//   ds_j  = p_j (dp_j - sum_l p_l dp_l)
//   dq_i  = sum_j ds_j k_j / sqrt(dh),     dk_j += ds_j q_i / sqrt(dh)
// Heads are split over threads; within a head the queries are visited in ascending order.
void oracle_swa_attention_backward(int64_t S, const double* q, const double* k, const double* v,
                                   const double* dout, int64_t nh, int64_t dh, int64_t w,
                                   double* dq, double* dk, double* dv, int threads) {
  const int64_t H = nh * dh;
  const double scale = 1.0 / std::sqrt((double)dh);
  for (int64_t i = 0; i < S * H; ++i) dq[i] = dk[i] = dv[i] = 0.0;
  for_row_ranges(nh, threads, [=](int64_t h0, int64_t h1) {
    std::vector<double> p(S > 0 ? S : 1), dp(S > 0 ? S : 1);
    for (int64_t head = h0; head < h1; ++head) {
      const int64_t off = head * dh;
      for (int64_t i = 0; i < S; ++i) {
        const int64_t j0 = std::max<int64_t>(0, i - w + 1);
        const double* qi = q + i * H + off;
        const double* doi = dout + i * H + off;
        double smax = -std::numeric_limits<double>::infinity();
        for (int64_t j = j0; j <= i; ++j) {
          double dot = 0.0;
          for (int64_t d = 0; d < dh; ++d) dot += qi[d] * k[j * H + off + d];
          p[j] = dot * scale;
          smax = std::max(smax, p[j]);
        }
        double denom = 0.0;
        for (int64_t j = j0; j <= i; ++j) {
          p[j] = std::exp(p[j] - smax);
          denom += p[j];
        }
        double pdp = 0.0;
        for (int64_t j = j0; j <= i; ++j) {
          p[j] /= denom;
          double dot = 0.0;
          for (int64_t d = 0; d < dh; ++d) dot += doi[d] * v[j * H + off + d];
          dp[j] = dot;
          pdp += p[j] * dp[j];
        }
        double* dqi = dq + i * H + off;
        for (int64_t j = j0; j <= i; ++j) {
          const double ds = p[j] * (dp[j] - pdp);
          for (int64_t d = 0; d < dh; ++d) {
            dqi[d] += ds * k[j * H + off + d] * scale;
            dk[j * H + off + d] += ds * qi[d] * scale;
            dv[j * H + off + d] += p[j] * doi[d];
          }
        }
      }
    }
  });
}

// Elementwise sum of n-vectors: out = a + b + c (the three terms of eq. (4)).
void oracle_add3(int64_t n, const double* a, const double* b, const double* c, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = a[i] + b[i] + c[i];
}

}  // extern "C"

// CPU oracle, C++17 + OpenMP: one top-k MoE FFN layer with SwiGLU experts,
// forward and backward, plus the e4m3 (FP8) variants.
//
// TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and the
// benchmark's CPU legs load this library.  The CUDA library never calls it,
// and it shares no code, header, table or helper with the CUDA sources.
//
// What it computes, and the passages it follows:
//
//  * Router and gating.  A gate network scores every expert for each token and
//    the k experts with the highest probability are chosen; their outputs are
//    summed with weights (DisagMoE, §2.1 "混合专家（MoE）结构"; the MegaScale-MoE
//    review lists the gate network as a component, §三 模型组件).  Reading:
//    l = x Wg + b, p = softmax over all E, the k largest logits (ties to the
//    lower expert id, slots in descending logit order), g_j = p_j / sum_sel p.
//  * Dispatch.  Token copies sorted by expert, then by source (MegaScale-MoE
//    digest §3.3 under Diagram C; the review's scatter that keeps memory
//    contiguous, §四 自适应EP通信策略详解).  On one GPU the source order is the
//    token order: a stable counting sort of the assignments a = t*k + j by
//    expert.  Optional capacity (the digest's per-GPU token dropping, §3.2 after
//    Figure 7: each expert keeps its first C assignments in assignment order)
//    and optional local expert range (the "scatter & drop" after the
//    all-gather, digest §3.2 Diagram B; review §四 step 2).
//  * Experts.  SwiGLU FFN per expert (review §三 核心公式; 训练流程 专家计算
//    GroupedGEMM): A = X W1, B = X W3, H = silu(A) * B, O = H W2.
//  * Combine.  y[t] = sum_j g[t,j] O[perm_dst[t*k+j]] (DisagMoE §2.1 weighted
//    sum; review 训练流程 Token聚合).
//  * Backward.  Written out as explicit operators (digest §3.3), by the chain
//    rule; FC2's weight gradient takes fc2_in (H) and the gradient of fc2_out
//    (review 选择性激活重计算).
//  * FP8.  Per-token e4m3 scales instead of per-tensor ones (review §三 创新点
//    FP8训练优化; digest §3.4).  Reading: one fp32 scale per activation row and
//    per weight output column (or output row for the data-gradient operand),
//    s = amax / 448 (1 for an all-zero vector), codes e4m3(v / s) with an fp32
//    division, exact code products summed, times s_row * s_col.
//
// Precision.  The record oracle ("_f32" entry points) takes the bf16 tensors
// as their 16-bit patterns (x, W1, W3, W2, dy: the bytes the layer receives)
// and Wg, b in fp32.  Every sum is accumulated in fp32 (float), in the plain
// loop order written below (each output's contraction index ascending), and
// every intermediate (A, B, H, O, dO, dH, dA, dB, dX) stays fp32: nothing is
// rounded to bf16 on the bf16 path.  The "_f64" entry points run the same
// templates in double on double inputs (any values), for finite-difference
// checks.  The code is compiled with -ffp-contract=off, so no multiply-add is
// fused and the results are the same on every host.
//
// Parallelism.  OpenMP splits only independent outputs (rows, or output rows
// of a weight gradient); every sum runs in one thread in the stated order, so
// the result does not depend on the thread count.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

using i64 = long long;

// ------------------------------------------------------------ number formats

inline float bf16_bits_to_float(uint16_t b) {
  uint32_t u = uint32_t(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// bfloat16 keeps the top 16 bits of an IEEE binary32; rounding to it is to
// the nearest value, ties to the even last kept bit.  NaN stays NaN.
inline float round_to_bf16(float v) {
  uint32_t u;
  std::memcpy(&u, &v, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) {
    u |= 0x00400000u;
    u &= 0xffff0000u;
  } else {
    uint32_t lsb = (u >> 16) & 1u;
    u = (u + 0x7fffu + lsb) & 0xffff0000u;
  }
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// e4m3 (OCP FP8 E4M3): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
// normal values 2^(e-7) * (1 + m/8) for e = 1..15 except e = 15, m = 7 (NaN),
// so the largest finite magnitude is 448; subnormals 2^-6 * m/8.  Rounding to
// it: nearest value, ties to an even mantissa; magnitudes above 448 saturate.
constexpr double kE4M3Max = 448.0;

double round_to_e4m3(double v) {
  if (std::isnan(v)) return v;
  double a = std::fabs(v);
  if (a == 0.0) return v;
  int ex = 0;
  std::frexp(a, &ex);                    // a = m * 2^ex, m in [0.5, 1)
  int binade = std::max(ex - 1, -6);     // values below 2^-6 use the subnormal spacing
  double step = std::ldexp(1.0, binade - 3);
  double r = std::nearbyint(a / step) * step;  // default rounding mode: ties to even
  r = std::min(r, kE4M3Max);
  return v < 0 ? -r : r;
}

// ----------------------------------------------------------- input readers

template <class S> inline S val(uint16_t b) { return S(bf16_bits_to_float(b)); }
template <class S> inline S val(float v) { return S(v); }
template <class S> inline S val(double v) { return S(v); }

template <class S> inline S exp_of(S z) { return S(std::exp(double(z))); }
template <class S> inline S sigmoid(S z) { return S(1) / (S(1) + exp_of<S>(-z)); }
// silu(z) = z * sigmoid(z), written as z / (1 + e^-z)
template <class S> inline S silu(S z) { return z / (S(1) + exp_of<S>(-z)); }

// -------------------------------------------------------------------- router

// l[t,e] = sum_i x[t,i] Wg[i,e] (+ b[e]); softmax over all E; the k largest
// logits (ties to the lower id), in descending order; g_j = p_j / sum_sel p.
template <class S, class X>
void route(i64 T, int h, int E, int k, const X* x, const S* Wg, const S* b, int32_t* idx,
           S* gates, S* logits) {
#pragma omp parallel
  {
    std::vector<int> ord(E);
    std::vector<S> p(E);
#pragma omp for schedule(static)
    for (i64 t = 0; t < T; ++t) {
      S* l = logits + t * E;
      for (int e = 0; e < E; ++e) l[e] = S(0);
      for (int i = 0; i < h; ++i) {
        const S xi = val<S>(x[t * h + i]);
        for (int e = 0; e < E; ++e) l[e] += xi * Wg[i64(i) * E + e];
      }
      if (b)
        for (int e = 0; e < E; ++e) l[e] += b[e];
      std::iota(ord.begin(), ord.end(), 0);
      std::stable_sort(ord.begin(), ord.end(), [&](int a, int c) { return l[a] > l[c]; });
      S m = l[ord[0]];
      S z = S(0);
      for (int e = 0; e < E; ++e) {
        p[e] = exp_of<S>(l[e] - m);
        z += p[e];
      }
      for (int e = 0; e < E; ++e) p[e] = p[e] / z;
      S zs = S(0);
      for (int j = 0; j < k; ++j) zs += p[ord[j]];
      for (int j = 0; j < k; ++j) {
        idx[t * k + j] = ord[j];
        gates[t * k + j] = p[ord[j]] / zs;
      }
    }
  }
}

// ------------------------------------------------------------------ dispatch

// Stable counting sort of the assignments a = 0..T*k-1 by expert, keeping
// only experts in [e_lo, e_hi) and, with capacity C >= 0, each expert's first
// C assignments in assignment order.  counts/offsets cover the local experts;
// perm_src[p] = a for the placed rows; perm_dst[a] = p, or -1 when dropped.
// An optional mask keep[a] = 0 drops assignment a up front (a token sample
// that must reproduce the drops of the whole batch).
// Returns the number of placed rows, or -1 for an expert id out of [0, E).
i64 dispatch(i64 T, int k, int E, const int32_t* idx, i64 capacity, int e_lo, int e_hi,
             int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* perm_dst,
             const uint8_t* keep = nullptr) {
  const i64 R = T * k;
  const int EL = e_hi - e_lo;
  std::vector<i64> kept(EL, 0);
  for (i64 a = 0; a < R; ++a) {
    const int e = idx[a];
    if (e < 0 || e >= E) return -1;
    perm_dst[a] = -1;
    if (e < e_lo || e >= e_hi) continue;
    if (keep && !keep[a]) continue;
    if (capacity >= 0 && kept[e - e_lo] >= capacity) continue;
    ++kept[e - e_lo];
    perm_dst[a] = 0;  // marked as kept; its row is assigned below
  }
  offsets[0] = 0;
  for (int e = 0; e < EL; ++e) {
    counts[e] = int32_t(kept[e]);
    offsets[e + 1] = offsets[e] + counts[e];
  }
  std::vector<i64> next(offsets, offsets + EL);
  for (i64 a = 0; a < R; ++a) {
    if (perm_dst[a] < 0) continue;
    const i64 p = next[idx[a] - e_lo]++;
    perm_dst[a] = int32_t(p);
    perm_src[p] = int32_t(a);
  }
  return offsets[EL];
}

// expert of every placed row: the e with offsets[e] <= p < offsets[e+1]
std::vector<int> row_experts(int E, const int32_t* offsets) {
  std::vector<int> ex(static_cast<size_t>(offsets[E]));
  for (int e = 0; e < E; ++e)
    for (i64 p = offsets[e]; p < offsets[e + 1]; ++p) ex[size_t(p)] = e;
  return ex;
}

// ------------------------------------------------------------------- experts

// Rows p of expert e (offsets[e] <= p < offsets[e+1]):
//   A[p,c] = sum_i X[p,i] W1[e,i,c],  B[p,c] = sum_i X[p,i] W3[e,i,c],
//   H = silu(A) * B,                  O[p,j] = sum_c H[p,c] W2[e,c,j].
template <class S, class W>
void expert_ffn_fwd(int h, int f, int E, const S* X, const int32_t* offsets, const W* W1,
                    const W* W3, const W* W2, S* A, S* B, S* H, S* O) {
  const std::vector<int> ex = row_experts(E, offsets);
  const i64 R = offsets[E];
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 p = 0; p < R; ++p) {
    const i64 e = ex[size_t(p)];
    S* a = A + p * f;
    S* bb = B + p * f;
    S* hh = H + p * f;
    S* o = O + p * h;
    for (int c = 0; c < f; ++c) a[c] = bb[c] = S(0);
    for (int i = 0; i < h; ++i) {
      const S xi = X[p * h + i];
      const W* w1 = W1 + (e * h + i) * f;
      const W* w3 = W3 + (e * h + i) * f;
      for (int c = 0; c < f; ++c) {
        a[c] += xi * val<S>(w1[c]);
        bb[c] += xi * val<S>(w3[c]);
      }
    }
    for (int c = 0; c < f; ++c) hh[c] = silu<S>(a[c]) * bb[c];
    for (int j = 0; j < h; ++j) o[j] = S(0);
    for (int c = 0; c < f; ++c) {
      const S hc = hh[c];
      const W* w2 = W2 + (e * f + c) * h;
      for (int j = 0; j < h; ++j) o[j] += hc * val<S>(w2[j]);
    }
  }
}

// y[t,:] = sum_{j<k} g[t,j] O[perm_dst[t*k+j], :], slots in order; a dropped
// slot (perm_dst = -1) adds nothing.
template <class S>
void combine(i64 T, int k, int h, const S* O, const S* gates, const int32_t* perm_dst, S* y) {
#pragma omp parallel for schedule(static)
  for (i64 t = 0; t < T; ++t) {
    S* yt = y + t * h;
    for (int c = 0; c < h; ++c) yt[c] = S(0);
    for (int j = 0; j < k; ++j) {
      const i64 p = perm_dst[t * k + j];
      if (p < 0) continue;
      const S g = gates[t * k + j];
      for (int c = 0; c < h; ++c) yt[c] += g * O[p * h + c];
    }
  }
}

// The expert backward given dO (the gradient of O), row by row:
//   dH[p,c] = sum_j dO[p,j] W2[e,c,j]
//   dA = dH * B * s * (1 + A (1 - s)), s = sigmoid(A)    (d silu(A)/dA = s (1 + A (1 - s)))
//   dB = dH * silu(A)
//   dX[p,i] = sum_c dA[p,c] W1[e,i,c] + sum_c dB[p,c] W3[e,i,c]  (one sum over both halves)
template <class S, class W>
void expert_rows_bwd(int h, int f, int E, const S* dO, const int32_t* offsets, const W* W1,
                     const W* W3, const W* W2, const S* A, const S* B, S* dA, S* dB, S* dX) {
  const std::vector<int> ex = row_experts(E, offsets);
  const i64 R = offsets[E];
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 p = 0; p < R; ++p) {
    const i64 e = ex[size_t(p)];
    const S* dop = dO + p * h;
    for (int c = 0; c < f; ++c) {
      const W* w2 = W2 + (e * f + c) * h;
      S dh = S(0);
      for (int j = 0; j < h; ++j) dh += dop[j] * val<S>(w2[j]);
      const S a = A[p * f + c];
      const S s = sigmoid<S>(a);
      dA[p * f + c] = dh * B[p * f + c] * s * (S(1) + a * (S(1) - s));
      dB[p * f + c] = dh * silu<S>(a);
    }
    for (int i = 0; i < h; ++i) {
      const W* w1 = W1 + (e * h + i) * f;
      const W* w3 = W3 + (e * h + i) * f;
      S acc = S(0);
      for (int c = 0; c < f; ++c) acc += dA[p * f + c] * val<S>(w1[c]);
      for (int c = 0; c < f; ++c) acc += dB[p * f + c] * val<S>(w3[c]);
      dX[p * h + i] = acc;
    }
  }
}

// The expert weight gradients, rows p ascending over each expert's rows:
//   dW2[e,c,j] = sum_p H[p,c] dO[p,j],  dW1[e,i,c] = sum_p X[p,i] dA[p,c],
//   dW3[e,i,c] = sum_p X[p,i] dB[p,c].   Experts without rows get zeros.
template <class S>
void expert_wgrads(int h, int f, int E, const S* dO, const S* X, const int32_t* offsets,
                   const S* H, const S* dA, const S* dB, S* dW1, S* dW3, S* dW2) {
#pragma omp parallel for schedule(dynamic, 4)
  for (i64 ei = 0; ei < i64(E) * h; ++ei) {
    const i64 e = ei / h, i = ei % h;
    S* w1 = dW1 + ei * f;
    S* w3 = dW3 + ei * f;
    for (int c = 0; c < f; ++c) w1[c] = w3[c] = S(0);
    for (i64 p = offsets[e]; p < offsets[e + 1]; ++p) {
      const S xv = X[p * h + i];
      for (int c = 0; c < f; ++c) {
        w1[c] += xv * dA[p * f + c];
        w3[c] += xv * dB[p * f + c];
      }
    }
  }
#pragma omp parallel for schedule(dynamic, 4)
  for (i64 ec = 0; ec < i64(E) * f; ++ec) {
    const i64 e = ec / f, c = ec % f;
    S* w2 = dW2 + ec * h;
    for (int j = 0; j < h; ++j) w2[j] = S(0);
    for (i64 p = offsets[e]; p < offsets[e + 1]; ++p) {
      const S hv = H[p * f + c];
      for (int j = 0; j < h; ++j) w2[j] += hv * dO[p * h + j];
    }
  }
}

template <class S, class W>
void expert_ffn_bwd(int h, int f, int E, const S* dO, const S* X, const int32_t* offsets,
                    const W* W1, const W* W3, const W* W2, const S* A, const S* B, const S* H,
                    S* dA, S* dB, S* dX, S* dW1, S* dW3, S* dW2) {
  expert_rows_bwd<S, W>(h, f, E, dO, offsets, W1, W3, W2, A, B, dA, dB, dX);
  expert_wgrads<S>(h, f, E, dO, X, offsets, H, dA, dB, dW1, dW3, dW2);
}

// Rows X [n,h] through one expert, with their gates g [n] and loss rows dY:
// o = FFN(X) [n,h], dg = <dY, o> [n] and dx = the expert's part of the row
// gradient, the rows backward of dO = g dY.  With dW1/dW3/dW2 non-null, also
// the expert's weight gradients from these rows alone.
template <class S, class W>
void expert_terms(i64 n, int h, int f, const S* X, const S* dY, const S* g, const W* W1e,
                  const W* W3e, const W* W2e, S* o, S* dg, S* dx, S* dW1, S* dW3, S* dW2) {
  const int32_t offsets[2] = {0, int32_t(n)};
  std::vector<S> A(size_t(n) * f), B(size_t(n) * f), H(size_t(n) * f), dO(size_t(n) * h);
  std::vector<S> dA(size_t(n) * f), dB(size_t(n) * f);
  expert_ffn_fwd<S, W>(h, f, 1, X, offsets, W1e, W3e, W2e, A.data(), B.data(), H.data(), o);
  for (i64 r = 0; r < n; ++r) {
    S acc = S(0);
    for (int j = 0; j < h; ++j) acc += dY[r * h + j] * o[r * h + j];
    dg[r] = acc;
    for (int j = 0; j < h; ++j) dO[size_t(r * h + j)] = g[r] * dY[r * h + j];
  }
  expert_rows_bwd<S, W>(h, f, 1, dO.data(), offsets, W1e, W3e, W2e, A.data(), B.data(),
                        dA.data(), dB.data(), dx);
  if (dW1 && dW3 && dW2)
    expert_wgrads<S>(h, f, 1, dO.data(), X, offsets, H.data(), dA.data(), dB.data(), dW1, dW3,
                     dW2);
}

// Gradient of the renormalised gates with respect to the selected logits.
// g = softmax over the k selected logits (the full-softmax denominator
// cancels), Jacobian g_j (delta_ij - g_i), so dl_j = g_j (dg_j - sum_i g_i dg_i);
// with sum_i g_i = 1 this is g_j sum_i g_i (dg_j - dg_i), evaluated in that
// form (no cancellation when one gate is near 1; exactly 0 for k = 1).
template <class S>
void router_bwd(i64 T, int k, const S* gates, const S* dg, S* dl_sel) {
#pragma omp parallel for schedule(static)
  for (i64 t = 0; t < T; ++t) {
    const S* g = gates + t * k;
    const S* d = dg + t * k;
    for (int j = 0; j < k; ++j) {
      S acc = S(0);
      for (int i = 0; i < k; ++i) acc += g[i] * (d[j] - d[i]);
      dl_sel[t * k + j] = g[j] * acc;
    }
  }
}

// ------------------------------------------------------------- whole layer

template <class S, class X>
void permute_rows(i64 R, int h, int k, const X* x, const int32_t* perm_src, S* x_perm) {
#pragma omp parallel for schedule(static)
  for (i64 p = 0; p < R; ++p) {
    const i64 t = perm_src[p] / k;
    for (int i = 0; i < h; ++i) x_perm[p * h + i] = val<S>(x[t * h + i]);
  }
}

template <class S, class X, class W>
i64 layer_fwd(i64 T, int h, int f, int E, int k, i64 capacity, const X* x, const S* Wg,
              const S* b, const W* W1, const W* W3, const W* W2, S* y, int32_t* idx, S* gates,
              S* logits, int32_t* counts, int32_t* offsets, int32_t* perm_src,
              int32_t* perm_dst, S* x_perm, S* A, S* B, S* H, S* O) {
  route<S, X>(T, h, E, k, x, Wg, b, idx, gates, logits);
  const i64 R = dispatch(T, k, E, idx, capacity, 0, E, counts, offsets, perm_src, perm_dst);
  if (R < 0) return R;
  permute_rows<S, X>(R, h, k, x, perm_src, x_perm);
  expert_ffn_fwd<S, W>(h, f, E, x_perm, offsets, W1, W3, W2, A, B, H, O);
  combine<S>(T, k, h, O, gates, perm_dst, y);
  return R;
}

// The token-side gradients, given dg (the gate gradients, [T*k]) and
// dX_perm (the expert backward's row gradients):
//   dl from router_bwd, scattered to [T, E] (0 off the selected experts);
//   dx[t] = sum_j dX_perm[perm_dst[t*k+j]] (kept slots) + sum_j dl[t,j] Wg[:, e_j];
//   dWg[i,e] = sum_t x[t,i] dl[t,e]  (t ascending).
template <class S, class X>
void token_grads(i64 T, int h, int E, int k, const X* x, const S* Wg, const int32_t* idx,
                 const S* gates, const int32_t* perm_dst, const S* dg, const S* dX_perm, S* dx,
                 S* dWg, S* dl) {
  std::vector<S> dl_sel(size_t(T * k));
  router_bwd<S>(T, k, gates, dg, dl_sel.data());
  for (i64 q = 0; q < T * E; ++q) dl[q] = S(0);
  for (i64 a = 0; a < T * k; ++a) dl[(a / k) * E + idx[a]] = dl_sel[size_t(a)];
#pragma omp parallel for schedule(static)
  for (i64 t = 0; t < T; ++t) {
    S* d = dx + t * h;
    for (int i = 0; i < h; ++i) d[i] = S(0);
    for (int j = 0; j < k; ++j) {
      const i64 p = perm_dst[t * k + j];
      if (p < 0) continue;
      for (int i = 0; i < h; ++i) d[i] += dX_perm[p * h + i];
    }
    for (int j = 0; j < k; ++j) {
      const S dlj = dl_sel[size_t(t * k + j)];
      const int e = idx[t * k + j];
      for (int i = 0; i < h; ++i) d[i] += dlj * Wg[i64(i) * E + e];
    }
  }
#pragma omp parallel for schedule(static)
  for (int i = 0; i < h; ++i) {
    S* w = dWg + i64(i) * E;
    for (int e = 0; e < E; ++e) w[e] = S(0);
    for (i64 t = 0; t < T; ++t) {
      const S xv = val<S>(x[t * h + i]);
      for (int e = 0; e < E; ++e) w[e] += xv * dl[t * E + e];
    }
  }
}

// dg[a] = <dy[t], O[p]> for a kept assignment a (t = a / k, p = perm_dst[a]),
// 0 for a dropped one.
template <class S, class X>
void gate_grads(i64 T, int h, int k, const X* dy, const int32_t* perm_dst, const S* O, S* dg) {
#pragma omp parallel for schedule(static)
  for (i64 a = 0; a < T * k; ++a) {
    const i64 p = perm_dst[a], t = a / k;
    S acc = S(0);
    if (p >= 0)
      for (int c = 0; c < h; ++c) acc += val<S>(dy[t * h + c]) * O[p * h + c];
    dg[a] = acc;
  }
}

// Gradients of L = <dy, y>: dO[p] = g[a] dy[t] (a = perm_src[p], t = a / k);
// dg; the expert backward; the token-side gradients.
template <class S, class X, class W>
void layer_bwd(i64 T, int h, int f, int E, int k, const X* x, const X* dy, const S* Wg,
               const W* W1, const W* W3, const W* W2, const int32_t* idx, const S* gates,
               const int32_t* offsets, const int32_t* perm_src, const int32_t* perm_dst,
               const S* x_perm, const S* A, const S* B, const S* H, const S* O, S* dx,
               S* dWg, S* dW1, S* dW3, S* dW2, S* dg, S* dl, S* dO, S* dA, S* dB, S* dX_perm) {
  const i64 R = offsets[E];
#pragma omp parallel for schedule(static)
  for (i64 p = 0; p < R; ++p) {
    const i64 a = perm_src[p], t = a / k;
    for (int c = 0; c < h; ++c) dO[p * h + c] = gates[a] * val<S>(dy[t * h + c]);
  }
  gate_grads<S, X>(T, h, k, dy, perm_dst, O, dg);
  expert_ffn_bwd<S, W>(h, f, E, dO, x_perm, offsets, W1, W3, W2, A, B, H, dA, dB, dX_perm, dW1,
                       dW3, dW2);
  token_grads<S, X>(T, h, E, k, x, Wg, idx, gates, perm_dst, dg, dX_perm, dx, dWg, dl);
}

// Columns c of dW1[e] and dW3[e] and rows c of dW2[e], for a set of nc
// columns c of the expert's width, from all of an expert's rows: X_e [n,h],
// their loss rows dY_e [n,h] and gates g_e [n] (dO_e = g_e dY_e).  Column c
// needs only A[:,c] = X_e W1[:,c], B[:,c] = X_e W3[:,c] and
// dH[:,c] = dO_e W2[c,:]^T.  The caller passes the selected weight columns
// as rows: W1c[q,:] = W1[:,c_q], W3c[q,:] = W3[:,c_q], W2r[q,:] = W2[c_q,:].
// Outputs: dW1t[q,:] = dW1[:,c_q], dW3t[q,:] = dW3[:,c_q], dW2r[q,:] = dW2[c_q,:].
template <class S, class W>
void expert_wgrad_columns(i64 n, int h, const S* X, const S* dY, const S* g, const W* W1c,
                          const W* W3c, const W* W2r, int nc, S* dW1t, S* dW3t, S* dW2r) {
  std::vector<S> da(size_t(n) * nc), db(size_t(n) * nc), hh(size_t(n) * nc);
  std::vector<S> dOv(size_t(n) * h);
  for (i64 r = 0; r < n; ++r)
    for (int i = 0; i < h; ++i) dOv[size_t(r * h + i)] = g[r] * dY[r * h + i];
  const S* dO = dOv.data();
#pragma omp parallel for schedule(static)
  for (i64 r = 0; r < n; ++r) {
    for (int q = 0; q < nc; ++q) {
      const W* w1 = W1c + i64(q) * h;
      const W* w3 = W3c + i64(q) * h;
      const W* w2 = W2r + i64(q) * h;
      S a = S(0), bb = S(0), dh = S(0);
      for (int i = 0; i < h; ++i) {
        a += X[r * h + i] * val<S>(w1[i]);
        bb += X[r * h + i] * val<S>(w3[i]);
        dh += dO[r * h + i] * val<S>(w2[i]);
      }
      const S s = sigmoid<S>(a);
      da[size_t(r * nc + q)] = dh * bb * s * (S(1) + a * (S(1) - s));
      db[size_t(r * nc + q)] = dh * silu<S>(a);
      hh[size_t(r * nc + q)] = silu<S>(a) * bb;
    }
  }
#pragma omp parallel for schedule(static)
  for (int q = 0; q < nc; ++q) {
    S* d1 = dW1t + i64(q) * h;
    S* d3 = dW3t + i64(q) * h;
    S* d2 = dW2r + i64(q) * h;
    for (int i = 0; i < h; ++i) d1[i] = d3[i] = d2[i] = S(0);
    for (i64 r = 0; r < n; ++r) {
      const S a = da[size_t(r * nc + q)], b = db[size_t(r * nc + q)];
      const S hv = hh[size_t(r * nc + q)];
      for (int i = 0; i < h; ++i) {
        d1[i] += X[r * h + i] * a;
        d3[i] += X[r * h + i] * b;
        d2[i] += hv * dO[r * h + i];
      }
    }
  }
}

// --------------------------------------------------------------------- FP8

// s = amax / 448 in fp32 (1 for an all-zero vector); codes e4m3(v / s), the
// division in fp32.
inline float scale_of(float amax) { return amax > 0.0f ? amax / float(kE4M3Max) : 1.0f; }
inline float code_of(float v, float s) { return float(round_to_e4m3(double(v / s))); }

void quantize_rows(i64 n, i64 m, const float* X, float* q, float* s) {
#pragma omp parallel for schedule(static)
  for (i64 r = 0; r < n; ++r) {
    float amax = 0.0f;
    for (i64 c = 0; c < m; ++c) amax = std::max(amax, std::fabs(X[r * m + c]));
    const float sc = scale_of(amax);
    s[r] = sc;
    for (i64 c = 0; c < m; ++c) q[r * m + c] = code_of(X[r * m + c], sc);
  }
}

// row r of X0 [n, m0] and row r of X1 [n, m1] share one scale (amax over both rows)
void quantize_rows_joint(i64 n, i64 m0, i64 m1, const float* X0, const float* X1, float* q0,
                         float* q1, float* s) {
#pragma omp parallel for schedule(static)
  for (i64 r = 0; r < n; ++r) {
    float amax = 0.0f;
    for (i64 c = 0; c < m0; ++c) amax = std::max(amax, std::fabs(X0[r * m0 + c]));
    for (i64 c = 0; c < m1; ++c) amax = std::max(amax, std::fabs(X1[r * m1 + c]));
    const float sc = scale_of(amax);
    s[r] = sc;
    for (i64 c = 0; c < m0; ++c) q0[r * m0 + c] = code_of(X0[r * m0 + c], sc);
    for (i64 c = 0; c < m1; ++c) q1[r * m1 + c] = code_of(X1[r * m1 + c], sc);
  }
}

// W [E, K, N]: one scale per (expert, output column n), amax over K
void quantize_cols(int E, i64 K, i64 N, const float* W, float* q, float* s) {
#pragma omp parallel for schedule(static)
  for (i64 en = 0; en < i64(E) * N; ++en) {
    const i64 e = en / N, n = en % N;
    float amax = 0.0f;
    for (i64 r = 0; r < K; ++r) amax = std::max(amax, std::fabs(W[(e * K + r) * N + n]));
    const float sc = scale_of(amax);
    s[en] = sc;
    for (i64 r = 0; r < K; ++r) q[(e * K + r) * N + n] = code_of(W[(e * K + r) * N + n], sc);
  }
}

// The expert forward on e4m3 codes: rows of X (x_perm) and of H one scale
// each; the columns of W1, W3, W2 one scale each.
//   A[p,c] = (sum_i Xq[p,i] W1q[e,i,c]) * sx[p] * s1[e,c]   (B likewise with W3)
//   H = bf16(silu(A) * B)   (the stored copy; its codes are made from it)
//   O[p,j] = (sum_c Hq[p,c] W2q[e,c,j]) * sh[p] * s2[e,j]
void expert_ffn_fwd_fp8(int h, int f, int E, const float* X, const int32_t* offsets,
                        const float* W1, const float* W3, const float* W2, float* A, float* B,
                        float* H, float* O, float* Xq, float* sx, float* Hq, float* sh,
                        float* W1q, float* s1, float* W3q, float* s3, float* W2q, float* s2) {
  const i64 R = offsets[E];
  quantize_rows(R, h, X, Xq, sx);
  quantize_cols(E, h, f, W1, W1q, s1);
  quantize_cols(E, h, f, W3, W3q, s3);
  quantize_cols(E, f, h, W2, W2q, s2);
  const std::vector<int> ex = row_experts(E, offsets);
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 p = 0; p < R; ++p) {
    const i64 e = ex[size_t(p)];
    std::vector<float> a(size_t(f), 0.0f), bb(size_t(f), 0.0f);
    for (int i = 0; i < h; ++i) {
      const float xq = Xq[p * h + i];
      for (int c = 0; c < f; ++c) {
        a[size_t(c)] += xq * W1q[(e * h + i) * f + c];
        bb[size_t(c)] += xq * W3q[(e * h + i) * f + c];
      }
    }
    for (int c = 0; c < f; ++c) {
      A[p * f + c] = a[size_t(c)] * sx[p] * s1[e * f + c];
      B[p * f + c] = bb[size_t(c)] * sx[p] * s3[e * f + c];
      H[p * f + c] = round_to_bf16(silu<float>(A[p * f + c]) * B[p * f + c]);
    }
  }
  quantize_rows(R, f, H, Hq, sh);
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 p = 0; p < R; ++p) {
    const i64 e = ex[size_t(p)];
    std::vector<float> o(size_t(h), 0.0f);
    for (int c = 0; c < f; ++c) {
      const float hq = Hq[p * f + c];
      for (int j = 0; j < h; ++j) o[size_t(j)] += hq * W2q[(e * f + c) * h + j];
    }
    for (int j = 0; j < h; ++j) O[p * h + j] = o[size_t(j)] * sh[p] * s2[e * h + j];
  }
}

// dX = dA W1e^T + dB W3e^T on e4m3 codes, one contraction over both halves:
// row r of dA and of dB share a scale; row i of W1e and of W3e ([h, f]) share
// a scale.  dX[r,i] = (sum_c dAq W1q + sum_c dBq W3q) * sa[r] * sw[i].
void fc1_dgrad_fp8(i64 n, int h, int f, const float* dA, const float* dB, const float* W1e,
                   const float* W3e, float* dX) {
  std::vector<float> aq(size_t(n) * f), bq(size_t(n) * f);
  std::vector<float> sa(static_cast<size_t>(n));
  std::vector<float> w1q(size_t(h) * f), w3q(size_t(h) * f);
  std::vector<float> sw(static_cast<size_t>(h));
  quantize_rows_joint(n, f, f, dA, dB, aq.data(), bq.data(), sa.data());
  quantize_rows_joint(h, f, f, W1e, W3e, w1q.data(), w3q.data(), sw.data());
#pragma omp parallel for schedule(static)
  for (i64 r = 0; r < n; ++r) {
    for (int i = 0; i < h; ++i) {
      float acc = 0.0f;
      for (int c = 0; c < f; ++c) acc += aq[size_t(r * f + c)] * w1q[size_t(i64(i) * f + c)];
      for (int c = 0; c < f; ++c) acc += bq[size_t(r * f + c)] * w3q[size_t(i64(i) * f + c)];
      dX[r * h + i] = acc * sa[size_t(r)] * sw[size_t(i)];
    }
  }
}

// The expert backward with the FC1 data gradient on e4m3 codes.  The layer
// keeps A, B, H in bf16, and the codes of dA and dB are made from the bf16
// values it stores, so here: A, B, H are rounded to bf16; dO is taken as
// given (the bf16 value of g * dy); dA and dB are rounded to bf16 and those
// copies feed both the FC1 dgrad codes and the weight gradients.
void expert_ffn_bwd_fp8(int h, int f, int E, const float* dO, const float* X,
                        const int32_t* offsets, const float* W1, const float* W3,
                        const float* W2, const float* A_in, const float* B_in,
                        const float* H_in, float* dA, float* dB, float* dX, float* dW1,
                        float* dW3, float* dW2) {
  const i64 R = offsets[E];
  std::vector<float> A(size_t(R) * f), B(size_t(R) * f), H(size_t(R) * f);
  for (i64 q = 0; q < R * f; ++q) {
    A[size_t(q)] = round_to_bf16(A_in[q]);
    B[size_t(q)] = round_to_bf16(B_in[q]);
    H[size_t(q)] = round_to_bf16(H_in[q]);
  }
  const std::vector<int> ex = row_experts(E, offsets);
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 p = 0; p < R; ++p) {
    const i64 e = ex[size_t(p)];
    for (int c = 0; c < f; ++c) {
      float dh = 0.0f;
      for (int j = 0; j < h; ++j) dh += dO[p * h + j] * W2[(e * f + c) * h + j];
      const float a = A[size_t(p * f + c)];
      const float s = sigmoid<float>(a);
      dA[p * f + c] = round_to_bf16(dh * B[size_t(p * f + c)] * s * (1.0f + a * (1.0f - s)));
      dB[p * f + c] = round_to_bf16(dh * silu<float>(a));
    }
  }
  for (int e = 0; e < E; ++e) {
    const i64 lo = offsets[e], n = offsets[e + 1] - lo;
    if (n > 0)
      fc1_dgrad_fp8(n, h, f, dA + lo * f, dB + lo * f, W1 + i64(e) * h * f,
                    W3 + i64(e) * h * f, dX + lo * h);
  }
#pragma omp parallel for schedule(dynamic, 4)
  for (i64 ei = 0; ei < i64(E) * h; ++ei) {
    const i64 e = ei / h, i = ei % h;
    for (int c = 0; c < f; ++c) dW1[ei * f + c] = dW3[ei * f + c] = 0.0f;
    for (i64 p = offsets[e]; p < offsets[e + 1]; ++p) {
      const float xv = X[p * h + i];
      for (int c = 0; c < f; ++c) {
        dW1[ei * f + c] += xv * dA[p * f + c];
        dW3[ei * f + c] += xv * dB[p * f + c];
      }
    }
  }
#pragma omp parallel for schedule(dynamic, 4)
  for (i64 ec = 0; ec < i64(E) * f; ++ec) {
    const i64 e = ec / f, c = ec % f;
    for (int j = 0; j < h; ++j) dW2[ec * h + j] = 0.0f;
    for (i64 p = offsets[e]; p < offsets[e + 1]; ++p) {
      const float hv = H[size_t(p * f + c)];
      for (int j = 0; j < h; ++j) dW2[ec * h + j] += hv * dO[p * h + j];
    }
  }
}

// The FP8 layer forward: route, dispatch, permute, expert_ffn_fwd_fp8, combine.
// The weights come as their bf16 patterns and are read as their exact values.
i64 layer_fwd_fp8(i64 T, int h, int f, int E, int k, i64 capacity, const uint16_t* x,
                  const float* Wg, const float* b, const uint16_t* W1b, const uint16_t* W3b,
                  const uint16_t* W2b, float* y, int32_t* idx, float* gates, float* logits,
                  int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* perm_dst,
                  float* x_perm, float* A, float* B, float* H, float* O, float* Xq, float* sx,
                  float* Hq, float* sh, float* W1q, float* s1, float* W3q, float* s3, float* W2q,
                  float* s2) {
  route<float, uint16_t>(T, h, E, k, x, Wg, b, idx, gates, logits);
  const i64 R = dispatch(T, k, E, idx, capacity, 0, E, counts, offsets, perm_src, perm_dst);
  if (R < 0) return R;
  permute_rows<float, uint16_t>(R, h, k, x, perm_src, x_perm);
  const i64 nw = i64(E) * h * f;
  std::vector<float> W1(static_cast<size_t>(nw)), W3(static_cast<size_t>(nw)),
      W2(static_cast<size_t>(nw));
  for (i64 q = 0; q < nw; ++q) {
    W1[size_t(q)] = bf16_bits_to_float(W1b[q]);
    W3[size_t(q)] = bf16_bits_to_float(W3b[q]);
    W2[size_t(q)] = bf16_bits_to_float(W2b[q]);
  }
  expert_ffn_fwd_fp8(h, f, E, x_perm, offsets, W1.data(), W3.data(), W2.data(), A, B, H, O, Xq,
                     sx, Hq, sh, W1q, s1, W3q, s3, W2q, s2);
  combine<float>(T, k, h, O, gates, perm_dst, y);
  return R;
}

// The FP8 layer backward: dO[p] = bf16(g[a] * dy[t]) (product in fp32, the
// layer stores dO in bf16); dg = <dy, O>; expert_ffn_bwd_fp8; the token-side
// gradients.
void layer_bwd_fp8(i64 T, int h, int f, int E, int k, const uint16_t* x, const uint16_t* dy,
                   const float* Wg, const uint16_t* W1b, const uint16_t* W3b,
                   const uint16_t* W2b, const int32_t* idx, const float* gates,
                   const int32_t* offsets, const int32_t* perm_src, const int32_t* perm_dst,
                   const float* x_perm, const float* A, const float* B, const float* H,
                   const float* O, float* dx, float* dWg, float* dW1, float* dW3, float* dW2,
                   float* dg, float* dl, float* dO, float* dA, float* dB, float* dX_perm) {
  const i64 R = offsets[E];
  for (i64 p = 0; p < R; ++p) {
    const i64 a = perm_src[p], t = a / k;
    for (int c = 0; c < h; ++c)
      dO[p * h + c] = round_to_bf16(gates[a] * bf16_bits_to_float(dy[t * h + c]));
  }
  gate_grads<float, uint16_t>(T, h, k, dy, perm_dst, O, dg);
  const i64 nw = i64(E) * h * f;
  std::vector<float> W1(static_cast<size_t>(nw)), W3(static_cast<size_t>(nw)),
      W2(static_cast<size_t>(nw));
  for (i64 q = 0; q < nw; ++q) {
    W1[size_t(q)] = bf16_bits_to_float(W1b[q]);
    W3[size_t(q)] = bf16_bits_to_float(W3b[q]);
    W2[size_t(q)] = bf16_bits_to_float(W2b[q]);
  }
  expert_ffn_bwd_fp8(h, f, E, dO, x_perm, offsets, W1.data(), W3.data(), W2.data(), A, B, H, dA,
                     dB, dX_perm, dW1, dW3, dW2);
  token_grads<float, uint16_t>(T, h, E, k, x, Wg, idx, gates, perm_dst, dg, dX_perm, dx, dWg,
                               dl);
}

}  // namespace

// =================================================================== C ABI
//
// Host pointers only; every array is caller-allocated, row-major and dense.
// Arrays of bf16 values are passed as their 16-bit patterns (uint16_t).
// R = T*k is the size of the assignment arrays; the permuted-row arrays
// (x_perm, A, B, H, O, dO, dA, dB, dX_perm) have room for T*k rows, of which
// the first offsets[E] are written.

extern "C" {

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_round_bf16(i64 n, const float* v, float* out) {
  for (i64 i = 0; i < n; ++i) out[i] = round_to_bf16(v[i]);
}

void oracle_round_e4m3(i64 n, const double* v, double* out) {
  for (i64 i = 0; i < n; ++i) out[i] = round_to_e4m3(v[i]);
}

// capacity < 0: dropless; keep may be NULL.  Returns the placed rows, -1 for
// a bad expert id.
i64 oracle_dispatch(i64 T, int k, int E, const int32_t* topk_idx, i64 capacity, int e_lo,
                    int e_hi, const uint8_t* keep, int32_t* counts, int32_t* offsets,
                    int32_t* perm_src, int32_t* perm_dst) {
  return dispatch(T, k, E, topk_idx, capacity, e_lo, e_hi, counts, offsets, perm_src, perm_dst,
                  keep);
}

void oracle_route_f32(i64 T, int h, int E, int k, const uint16_t* x, const float* Wg,
                      const float* b, int32_t* idx, float* gates, float* logits) {
  route<float, uint16_t>(T, h, E, k, x, Wg, b, idx, gates, logits);
}
void oracle_route_f64(i64 T, int h, int E, int k, const double* x, const double* Wg,
                      const double* b, int32_t* idx, double* gates, double* logits) {
  route<double, double>(T, h, E, k, x, Wg, b, idx, gates, logits);
}

void oracle_expert_ffn_fwd_f32(int h, int f, int E, const float* X, const int32_t* offsets,
                               const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                               float* A, float* B, float* H, float* O) {
  expert_ffn_fwd<float, uint16_t>(h, f, E, X, offsets, W1, W3, W2, A, B, H, O);
}
void oracle_expert_ffn_fwd_f64(int h, int f, int E, const double* X, const int32_t* offsets,
                               const double* W1, const double* W3, const double* W2, double* A,
                               double* B, double* H, double* O) {
  expert_ffn_fwd<double, double>(h, f, E, X, offsets, W1, W3, W2, A, B, H, O);
}

void oracle_combine_f32(i64 T, int k, int h, const float* O, const float* gates,
                        const int32_t* perm_dst, float* y) {
  combine<float>(T, k, h, O, gates, perm_dst, y);
}
void oracle_combine_f64(i64 T, int k, int h, const double* O, const double* gates,
                        const int32_t* perm_dst, double* y) {
  combine<double>(T, k, h, O, gates, perm_dst, y);
}

void oracle_expert_ffn_bwd_f32(int h, int f, int E, const float* dO, const float* X,
                               const int32_t* offsets, const uint16_t* W1, const uint16_t* W3,
                               const uint16_t* W2, const float* A, const float* B,
                               const float* H, float* dA, float* dB, float* dX, float* dW1,
                               float* dW3, float* dW2) {
  expert_ffn_bwd<float, uint16_t>(h, f, E, dO, X, offsets, W1, W3, W2, A, B, H, dA, dB, dX, dW1,
                                  dW3, dW2);
}
void oracle_expert_ffn_bwd_f64(int h, int f, int E, const double* dO, const double* X,
                               const int32_t* offsets, const double* W1, const double* W3,
                               const double* W2, const double* A, const double* B,
                               const double* H, double* dA, double* dB, double* dX,
                               double* dW1, double* dW3, double* dW2) {
  expert_ffn_bwd<double, double>(h, f, E, dO, X, offsets, W1, W3, W2, A, B, H, dA, dB, dX, dW1,
                                 dW3, dW2);
}

void oracle_router_bwd_f32(i64 T, int k, const float* gates, const float* dg, float* dl_sel) {
  router_bwd<float>(T, k, gates, dg, dl_sel);
}
void oracle_router_bwd_f64(i64 T, int k, const double* gates, const double* dg,
                           double* dl_sel) {
  router_bwd<double>(T, k, gates, dg, dl_sel);
}

i64 oracle_layer_fwd_f32(i64 T, int h, int f, int E, int k, i64 capacity, const uint16_t* x,
                         const float* Wg, const float* b, const uint16_t* W1,
                         const uint16_t* W3, const uint16_t* W2, float* y, int32_t* idx,
                         float* gates, float* logits, int32_t* counts, int32_t* offsets,
                         int32_t* perm_src, int32_t* perm_dst, float* x_perm, float* A, float* B,
                         float* H, float* O) {
  return layer_fwd<float, uint16_t, uint16_t>(T, h, f, E, k, capacity, x, Wg, b, W1, W3, W2, y,
                                              idx, gates, logits, counts, offsets, perm_src,
                                              perm_dst, x_perm, A, B, H, O);
}
i64 oracle_layer_fwd_f64(i64 T, int h, int f, int E, int k, i64 capacity, const double* x,
                         const double* Wg, const double* b, const double* W1, const double* W3,
                         const double* W2, double* y, int32_t* idx, double* gates,
                         double* logits, int32_t* counts, int32_t* offsets, int32_t* perm_src,
                         int32_t* perm_dst, double* x_perm, double* A, double* B, double* H,
                         double* O) {
  return layer_fwd<double, double, double>(T, h, f, E, k, capacity, x, Wg, b, W1, W3, W2, y, idx,
                                           gates, logits, counts, offsets, perm_src, perm_dst,
                                           x_perm, A, B, H, O);
}

void oracle_layer_bwd_f32(i64 T, int h, int f, int E, int k, const uint16_t* x,
                          const uint16_t* dy, const float* Wg, const uint16_t* W1,
                          const uint16_t* W3, const uint16_t* W2, const int32_t* idx,
                          const float* gates, const int32_t* offsets, const int32_t* perm_src,
                          const int32_t* perm_dst, const float* x_perm, const float* A,
                          const float* B, const float* H, const float* O, float* dx, float* dWg,
                          float* dW1, float* dW3, float* dW2, float* dg, float* dl, float* dO,
                          float* dA, float* dB, float* dX_perm) {
  layer_bwd<float, uint16_t, uint16_t>(T, h, f, E, k, x, dy, Wg, W1, W3, W2, idx, gates, offsets,
                                       perm_src, perm_dst, x_perm, A, B, H, O, dx, dWg, dW1, dW3,
                                       dW2, dg, dl, dO, dA, dB, dX_perm);
}
void oracle_layer_bwd_f64(i64 T, int h, int f, int E, int k, const double* x, const double* dy,
                          const double* Wg, const double* W1, const double* W3,
                          const double* W2, const int32_t* idx, const double* gates,
                          const int32_t* offsets, const int32_t* perm_src,
                          const int32_t* perm_dst, const double* x_perm, const double* A,
                          const double* B, const double* H, const double* O, double* dx,
                          double* dWg, double* dW1, double* dW3, double* dW2, double* dg,
                          double* dl, double* dO, double* dA, double* dB, double* dX_perm) {
  layer_bwd<double, double, double>(T, h, f, E, k, x, dy, Wg, W1, W3, W2, idx, gates, offsets,
                                    perm_src, perm_dst, x_perm, A, B, H, O, dx, dWg, dW1, dW3,
                                    dW2, dg, dl, dO, dA, dB, dX_perm);
}

void oracle_expert_wgrad_columns_f32(i64 n, int h, const float* X, const float* dY,
                                     const float* g, const uint16_t* W1c, const uint16_t* W3c,
                                     const uint16_t* W2r, int nc, float* dW1t, float* dW3t,
                                     float* dW2r) {
  expert_wgrad_columns<float, uint16_t>(n, h, X, dY, g, W1c, W3c, W2r, nc, dW1t, dW3t, dW2r);
}
void oracle_expert_wgrad_columns_f64(i64 n, int h, const double* X, const double* dY,
                                     const double* g, const double* W1c, const double* W3c,
                                     const double* W2r, int nc, double* dW1t, double* dW3t,
                                     double* dW2r) {
  expert_wgrad_columns<double, double>(n, h, X, dY, g, W1c, W3c, W2r, nc, dW1t, dW3t, dW2r);
}

void oracle_quantize_rows_e4m3(i64 n, i64 m, const float* X, float* q, float* s) {
  quantize_rows(n, m, X, q, s);
}
void oracle_quantize_rows_joint_e4m3(i64 n, i64 m0, i64 m1, const float* X0, const float* X1,
                                     float* q0, float* q1, float* s) {
  quantize_rows_joint(n, m0, m1, X0, X1, q0, q1, s);
}
void oracle_quantize_cols_e4m3(int E, i64 K, i64 N, const float* W, float* q, float* s) {
  quantize_cols(E, K, N, W, q, s);
}
void oracle_expert_ffn_fwd_fp8(int h, int f, int E, const float* X, const int32_t* offsets,
                               const float* W1, const float* W3, const float* W2, float* A,
                               float* B, float* H, float* O, float* Xq, float* sx, float* Hq,
                               float* sh, float* W1q, float* s1, float* W3q, float* s3,
                               float* W2q, float* s2) {
  expert_ffn_fwd_fp8(h, f, E, X, offsets, W1, W3, W2, A, B, H, O, Xq, sx, Hq, sh, W1q, s1, W3q,
                     s3, W2q, s2);
}
void oracle_fc1_dgrad_fp8(i64 n, int h, int f, const float* dA, const float* dB,
                          const float* W1e, const float* W3e, float* dX) {
  fc1_dgrad_fp8(n, h, f, dA, dB, W1e, W3e, dX);
}
void oracle_expert_ffn_bwd_fp8(int h, int f, int E, const float* dO, const float* X,
                               const int32_t* offsets, const float* W1, const float* W3,
                               const float* W2, const float* A, const float* B, const float* H,
                               float* dA, float* dB, float* dX, float* dW1, float* dW3,
                               float* dW2) {
  expert_ffn_bwd_fp8(h, f, E, dO, X, offsets, W1, W3, W2, A, B, H, dA, dB, dX, dW1, dW3, dW2);
}

i64 oracle_layer_fwd_fp8(i64 T, int h, int f, int E, int k, i64 capacity, const uint16_t* x,
                         const float* Wg, const float* b, const uint16_t* W1,
                         const uint16_t* W3, const uint16_t* W2, float* y, int32_t* idx,
                         float* gates, float* logits, int32_t* counts, int32_t* offsets,
                         int32_t* perm_src, int32_t* perm_dst, float* x_perm, float* A, float* B,
                         float* H, float* O, float* Xq, float* sx, float* Hq, float* sh,
                         float* W1q, float* s1, float* W3q, float* s3, float* W2q, float* s2) {
  return layer_fwd_fp8(T, h, f, E, k, capacity, x, Wg, b, W1, W3, W2, y, idx, gates, logits,
                       counts, offsets, perm_src, perm_dst, x_perm, A, B, H, O, Xq, sx, Hq, sh,
                       W1q, s1, W3q, s3, W2q, s2);
}
void oracle_layer_bwd_fp8(i64 T, int h, int f, int E, int k, const uint16_t* x,
                          const uint16_t* dy, const float* Wg, const uint16_t* W1,
                          const uint16_t* W3, const uint16_t* W2, const int32_t* idx,
                          const float* gates, const int32_t* offsets, const int32_t* perm_src,
                          const int32_t* perm_dst, const float* x_perm, const float* A,
                          const float* B, const float* H, const float* O, float* dx, float* dWg,
                          float* dW1, float* dW3, float* dW2, float* dg, float* dl, float* dO,
                          float* dA, float* dB, float* dX_perm) {
  layer_bwd_fp8(T, h, f, E, k, x, dy, Wg, W1, W3, W2, idx, gates, offsets, perm_src, perm_dst,
                x_perm, A, B, H, O, dx, dWg, dW1, dW3, dW2, dg, dl, dO, dA, dB, dX_perm);
}

void oracle_permute_rows_f32(i64 R, int h, int k, const uint16_t* x, const int32_t* perm_src,
                             float* x_perm) {
  permute_rows<float, uint16_t>(R, h, k, x, perm_src, x_perm);
}

void oracle_token_grads_f32(i64 T, int h, int E, int k, const uint16_t* x, const float* Wg,
                            const int32_t* idx, const float* gates, const int32_t* perm_dst,
                            const float* dg, const float* dX_perm, float* dx, float* dWg,
                            float* dl) {
  token_grads<float, uint16_t>(T, h, E, k, x, Wg, idx, gates, perm_dst, dg, dX_perm, dx, dWg, dl);
}

// dW1, dW3 [h,f] and dW2 [f,h] may be NULL (rows only)
void oracle_expert_terms_f32(i64 n, int h, int f, const float* X, const float* dY,
                             const float* g, const uint16_t* W1e, const uint16_t* W3e,
                             const uint16_t* W2e, float* o, float* dg, float* dx, float* dW1,
                             float* dW3, float* dW2) {
  expert_terms<float, uint16_t>(n, h, f, X, dY, g, W1e, W3e, W2e, o, dg, dx, dW1, dW3, dW2);
}
void oracle_expert_terms_f64(i64 n, int h, int f, const double* X, const double* dY,
                             const double* g, const double* W1e, const double* W3e,
                             const double* W2e, double* o, double* dg, double* dx, double* dW1,
                             double* dW3, double* dW2) {
  expert_terms<double, double>(n, h, f, X, dY, g, W1e, W3e, W2e, o, dg, dx, dW1, dW3, dW2);
}

void oracle_token_grads_f64(i64 T, int h, int E, int k, const double* x, const double* Wg,
                            const int32_t* idx, const double* gates, const int32_t* perm_dst,
                            const double* dg, const double* dX_perm, double* dx, double* dWg,
                            double* dl) {
  token_grads<double, double>(T, h, E, k, x, Wg, idx, gates, perm_dst, dg, dX_perm, dx, dWg, dl);
}

void oracle_permute_rows_f64(i64 R, int h, int k, const double* x, const int32_t* perm_src,
                             double* x_perm) {
  permute_rows<double, double>(R, h, k, x, perm_src, x_perm);
}

}  // extern "C"

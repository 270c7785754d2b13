// Row-wise and small kernels of the GRPO loss path: group advantages, the
// row plan (per-sequence counts and the list of 128-row blocks holding a
// valid token), the per-token loss terms with deterministic float64
// reductions, the backward coefficients, the W transpose and fills.
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace grpo {

namespace {

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------- advantages
// Group-relative advantages: several answers per prompt are scored and the
// advantage comes from the rewards statistically (aibit.im GRPO blog, GRPO
// section; zjt100.com translation of the Unsloth GRPO blog, "GRPO 的数学和
// 发现的问题": A is the advantage after all reward functions). The pages
// print no formula; the reading is A = (r - mean_g) / (std_g + eps).
// One warp per group of G contiguous rewards; mean and std in float64.
__global__ void k_advantages(const float* __restrict__ r, int B, int G, float eps, int unbiased,
                             float* __restrict__ adv) {
  const int grp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (grp >= B / G) return;
  const float* rg = r + static_cast<int64_t>(grp) * G;
  double s = 0.0;
  for (int i = lane; i < G; i += 32) s += static_cast<double>(rg[i]);
  const double mean = warp_sum_d(s) / G;
  double v = 0.0;
  for (int i = lane; i < G; i += 32) {
    const double dd = static_cast<double>(rg[i]) - mean;
    v += dd * dd;
  }
  const double sd = sqrt(warp_sum_d(v) / (G - unbiased));
  const double den = sd + static_cast<double>(eps);
  for (int i = lane; i < G; i += 32)
    adv[static_cast<int64_t>(grp) * G + i] =
        static_cast<float>((static_cast<double>(rg[i]) - mean) / den);
}

// --------------------------------------------------------------- convert
__global__ void k_convert_bf16(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                               int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i * 4 < n;
       i += stride) {
    const int64_t e = i * 4;
    if (e + 4 <= n) {
      const float4 v = *reinterpret_cast<const float4*>(src + e);
      uint2 o;
      o.x = pack_bf16x2(v.x, v.y);
      o.y = pack_bf16x2(v.z, v.w);
      *reinterpret_cast<uint2*>(dst + e) = o;
    } else {
      for (int64_t k = e; k < n; ++k) dst[k] = __float2bfloat16_rn(src[k]);
    }
  }
}

// ------------------------------------------------------------- seq count
// The loss scores completion tokens (Unsloth "grpo-long-context" page,
// flattened sequence chunking: hidden states and completion ids are passed
// together); masked positions are excluded.
// One CTA per sequence: cnt_b = number of valid tokens; valid tokens whose id
// is outside [0, V) raise the bad-token bit.
__global__ void k_seq_count(const uint8_t* __restrict__ mask, const int32_t* __restrict__ ids,
                            int T, int64_t V, int* __restrict__ cnt, uint32_t* err) {
  __shared__ int wsum[32];
  const int b = blockIdx.x;
  const int64_t r0 = static_cast<int64_t>(b) * T;
  int c = 0;
  bool bad = false;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    if (mask[r0 + t]) {
      ++c;
      const int32_t y = ids[r0 + t];
      bad |= (y < 0) || (static_cast<int64_t>(y) >= V);
    }
  }
  if (bad) atomicOr(err, ERRBIT_BAD_TOKEN);
  c = warp_sum_i(c);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x < 32) {
    int v = threadIdx.x < (blockDim.x >> 5) ? wsum[threadIdx.x] : 0;
    v = warp_sum_i(v);
    if (threadIdx.x == 0) cnt[b] = v;
  }
}

// ------------------------------------------------------------ block plan
// Single CTA of 1024 threads: flag each 128-row block that holds a valid
// token, then compact the flagged blocks in order (block-wide scan).
__global__ void __launch_bounds__(1024) k_block_plan(const uint8_t* __restrict__ mask, int64_t N,
                                                     int nblk, int* __restrict__ blk,
                                                     int* __restrict__ inv, int* nblk_dev) {
  __shared__ int wtot[32];
  __shared__ int base;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) base = 0;
  __syncthreads();
  const bool aligned = (reinterpret_cast<uintptr_t>(mask) & 15) == 0;
  for (int k0 = 0; k0 < nblk; k0 += 1024) {
    const int k = k0 + threadIdx.x;
    int flag = 0;
    if (k < nblk) {
      const int64_t r0 = static_cast<int64_t>(k) * kBM;
      const int64_t r1 = min(N, r0 + kBM);
      if (aligned && r1 - r0 == kBM) {
        const uint4* p = reinterpret_cast<const uint4*>(mask + r0);
        uint32_t acc = 0;
#pragma unroll
        for (int i = 0; i < kBM / 16; ++i) {
          const uint4 v = p[i];
          acc |= v.x | v.y | v.z | v.w;
        }
        flag = acc != 0;
      } else {
        for (int64_t r = r0; r < r1; ++r) flag |= mask[r] != 0;
      }
    }
    // inclusive scan of flag across the CTA
    int x = flag;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = wtot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      wtot[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const int excl = x - flag + (warp > 0 ? wtot[warp - 1] : 0);
    if (k < nblk) {
      inv[k] = flag ? base + excl : -1;
      if (flag) blk[base + excl] = k;
    }
    __syncthreads();
    if (threadIdx.x == 0) base += wtot[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) *nblk_dev = base;
}

// ------------------------------------------------------------ fwd finish
// The objective of the zjt100.com page, "GRPO 的数学和发现的问题": reverse KL
// with Q the trained model and P the frozen reference, beta = 0.04, the
// estimator exp(x) - x - 1 (x = p - q) with no extra Q factor, and the
// exp(q - q.detach()) * A term, whose value is 1. The kl_mode variants read
// the page's four experiments (same section).
// Merge the vocab-slice partials into each row's logsumexp, form q, p, the
// KL estimator and the weighted loss terms. Per-CTA float64 partial sums
// (sum w*A, sum w*KL, sum m*KL) go to `partials` for a fixed-order final sum.
// Per-token KL term of the selected mode, x = p - q (see grpo_problem.kl_mode).
__device__ __forceinline__ float kl_term(float q, float x, int kl_mode) {
  const float k3 = __fsub_rn(expm1f(x), x);
  if (kl_mode == 2) return __fmul_rn(expf(q), k3);
  if (kl_mode == 3) return __fsub_rn(__fmul_rn(x, expf(x)), expm1f(x));
  return k3;
}

// Rounding is spelled out (__fmaf_rn, __fadd_rn, __fmul_rn) so that every
// inlined copy computes bit-identical results: equal policy and reference
// rows then give exactly x = p - q = 0.
__device__ __noinline__ float merge_lse(const float2* p, int n_vs) {
  float M = -INFINITY;
  for (int v = 0; v < n_vs; ++v) M = fmaxf(M, p[static_cast<int64_t>(v) * kBM].x);
  float S = 0.f;
  for (int v = 0; v < n_vs; ++v) {
    const float2 e = p[static_cast<int64_t>(v) * kBM];
    S = __fmaf_rn(e.y, exp2f(__fsub_rn(e.x, M)), S);
  }
  return __fmul_rn(__fadd_rn(M, log2f(S)), 0.69314718055994531f);
}

// token_level: the weights are 1 here and the final sum is divided by the
// number of valid tokens. ref_given: p is read from logp_ref (and logp_ref is
// not written).
__global__ void k_fwd_finish(const int* __restrict__ inv, const uint8_t* __restrict__ mask,
                             const int* __restrict__ cnt, const float* __restrict__ adv,
                             const float* __restrict__ zy, const float2* __restrict__ part,
                             int nblk_max, int n_vs, int64_t N, int B, int T, int token_level,
                             int ref_given, int kl_mode, float* __restrict__ logp_pol,
                             float* __restrict__ logp_ref, float* __restrict__ lse_pol,
                             double* __restrict__ partials) {
  __shared__ double red[3][32];
  double sa = 0.0, sk = 0.0, sm = 0.0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < N;
       n += stride) {
    const int k = static_cast<int>(n / kBM);
    const int j = inv[k];
    float lp = 0.f, lr = 0.f, ls = 0.f;
    if (j >= 0) {
      const int r = static_cast<int>(n - static_cast<int64_t>(k) * kBM);
      const float2* pp = part + (static_cast<int64_t>(j) * n_vs) * kBM + r;
      const float2* pr = part + ((static_cast<int64_t>(nblk_max) + j) * n_vs) * kBM + r;
      ls = merge_lse(pp, n_vs);
      if (mask[n]) {
        const float q = __fsub_rn(zy[n], ls);
        const float p = ref_given ? logp_ref[n] : __fsub_rn(zy[N + n], merge_lse(pr, n_vs));
        lp = q;
        lr = p;
        const float x = __fsub_rn(p, q);
        const float kl = kl_term(q, x, kl_mode);
        const int b = static_cast<int>(n / T);
        const double w =
            token_level ? 1.0 : 1.0 / (static_cast<double>(B) * max(cnt[b], 1));
        sa += w * static_cast<double>(adv[b]);
        sk += w * static_cast<double>(kl);
        sm += static_cast<double>(kl);
      }
    }
    logp_pol[n] = lp;
    if (!ref_given) logp_ref[n] = lr;
    lse_pol[n] = ls;
  }
  sa = warp_sum_d(sa);
  sk = warp_sum_d(sk);
  sm = warp_sum_d(sm);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    red[0][warp] = sa;
    red[1][warp] = sk;
    red[2][warp] = sm;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    double a = lane < nw ? red[0][lane] : 0.0;
    double b = lane < nw ? red[1][lane] : 0.0;
    double c = lane < nw ? red[2][lane] : 0.0;
    a = warp_sum_d(a);
    b = warp_sum_d(b);
    c = warp_sum_d(c);
    if (lane == 0) {
      partials[3 * blockIdx.x + 0] = a;
      partials[3 * blockIdx.x + 1] = b;
      partials[3 * blockIdx.x + 2] = c;
    }
  }
}

// Single warp: fixed-order sum of the per-CTA partials.
__global__ void k_fwd_reduce(const double* __restrict__ partials, int nparts,
                             const int* __restrict__ cnt, int B, float beta, int token_level,
                             float* loss, float* kl_mean) {
  const int lane = threadIdx.x;
  double a = 0.0, k = 0.0, m = 0.0, c = 0.0;
  for (int i = lane; i < nparts; i += 32) {
    a += partials[3 * i + 0];
    k += partials[3 * i + 1];
    m += partials[3 * i + 2];
  }
  for (int i = lane; i < B; i += 32) c += static_cast<double>(cnt[i]);
  a = warp_sum_d(a);
  k = warp_sum_d(k);
  m = warp_sum_d(m);
  c = warp_sum_d(c);
  if (lane == 0) {
    const double l = -a + static_cast<double>(beta) * k;
    *loss = static_cast<float>(token_level ? l / (c > 1.0 ? c : 1.0) : l);
    if (kl_mean) *kl_mean = c > 0.0 ? static_cast<float>(m / c) : 0.f;
  }
}

// -------------------------------------------------------- bwd coefficient
// The derivative of the per-token loss with respect to q (same page and
// section): the detached factor passes A * dq, and d/dq of the estimator is
// 1 - exp(x). So c_n = -dloss/dq_n, and dZ_n = c_n (softmax(z_n) - onehot).
// c_n = g * w_n * (A_b + beta * (exp(p - q) - 1)) at valid rows, 0 elsewhere.
// Token level: w_n = 1 / max(sum_b cnt_b, 1), the total formed per CTA.
__global__ void k_bwd_coef(const uint8_t* __restrict__ mask, const int* __restrict__ cnt,
                           const float* __restrict__ adv, const float* __restrict__ logp_pol,
                           const float* __restrict__ logp_ref, int64_t N, int B, int T,
                           float beta, float grad, int token_level, int kl_mode,
                           float* __restrict__ coef) {
  __shared__ int64_t s_tot[32];
  double w_tok = 0.0;
  if (token_level) {
    int64_t t = 0;
    for (int i = threadIdx.x; i < B; i += blockDim.x) t += cnt[i];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if ((threadIdx.x & 31) == 0) s_tot[threadIdx.x >> 5] = t;
    __syncthreads();
    int64_t tot = 0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) tot += s_tot[i];
    w_tok = 1.0 / static_cast<double>(tot > 1 ? tot : 1);
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < N;
       n += stride) {
    float c = 0.f;
    if (mask[n]) {
      const int b = static_cast<int>(n / T);
      const double w =
          token_level ? w_tok : 1.0 / (static_cast<double>(B) * max(cnt[b], 1));
      // c = g w (a - beta dKL/dq); a = A_b except without the detach
      const float q = logp_pol[n];
      const float x = logp_ref[n] - q;
      float mdk;  // -dKL/dq
      if (kl_mode == 2)
        mdk = x * expf(q);
      else if (kl_mode == 3)
        mdk = x * expf(x);
      else
        mdk = expm1f(x);
      const double a = kl_mode == 1 ? 0.0 : static_cast<double>(adv[b]);
      c = static_cast<float>(static_cast<double>(grad) * w *
                             (a + static_cast<double>(beta) * static_cast<double>(mdk)));
    }
    coef[n] = c;
  }
}

// ------------------------------------------------------------- transpose
// One element of a matrix of element type ELT as float: bf16 and float32 as
// stored; e4m3 decoded exactly and multiplied by its row's scale.
template <int ELT>
__device__ __forceinline__ float load_elt(const void* base, const float* row_scale, int64_t r,
                                          int64_t i) {
  if constexpr (ELT == ELT_F32) {
    return static_cast<const float*>(base)[i];
  } else if constexpr (ELT == ELT_BF16) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
  } else {
    __nv_fp8_e4m3 v;
    v.__x = static_cast<const uint8_t*>(base)[i];
    return static_cast<float>(v) * row_scale[r];
  }
}

// Wt[c][r] = bf16(W[r][c]) for W [V, d], 32x32 tiles.
template <int ELT>
__global__ void k_transpose_w(const void* __restrict__ W, const float* __restrict__ w_scale,
                              int64_t V, int64_t d, __nv_bfloat16* __restrict__ Wt,
                              int64_t ldwt) {
  __shared__ float tile[32][33];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    float v = 0.f;
    if (r < V && c < d) v = load_elt<ELT>(W, w_scale, r, r * d + c);
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (c < d && r < V) Wt[c * ldwt + r] = __float2bfloat16_rn(tile[threadIdx.x][i]);
  }
}

// bf16 W [V, d] -> Wt [d, ldwt] in 64 x 64 tiles with 16-byte accesses on
// both sides (d and ldwt multiples of 8; W and Wt 16-byte aligned). A
// thread moves 8 elements per access: rows of the tile are read as 8 chunks
// of 16 bytes by 8 consecutive threads, and written back the same way as
// rows of Wt. The tile is held as float with a 65-word row pitch, so the
// row-wise writes and the column-wise reads of a warp (4 rows x 8 chunks)
// fall in 32 different banks. Columns of Wt past V (up to ldwt) get zeros.
constexpr int kTT = 64;  // tile edge of the vectorized transposes
__global__ void __launch_bounds__(256) k_transpose_w_bf16(const __nv_bfloat16* __restrict__ W,
                                                          int64_t V, int64_t d,
                                                          __nv_bfloat16* __restrict__ Wt,
                                                          int64_t ldwt) {
  __shared__ float tile[kTT][kTT + 1];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTT;  // rows of W
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kTT;  // columns of W
  const int i = threadIdx.x >> 3, j = threadIdx.x & 7;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int rr = i + 32 * p;
    const int64_t r = r0 + rr, c = c0 + 8 * j;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < V && c < d) v = *reinterpret_cast<const uint4*>(W + r * d + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      tile[rr][8 * j + 2 * k] = __uint_as_float(w[k] << 16);
      tile[rr][8 * j + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int cc = i + 32 * p;
    const int64_t c = c0 + cc, r = r0 + 8 * j;
    if (c < d && r < ldwt) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = __float_as_uint(tile[8 * j + 2 * k][cc]) >> 16;
        const uint32_t hi = __float_as_uint(tile[8 * j + 2 * k + 1][cc]) & 0xFFFF0000u;
        w[k] = lo | hi;
      }
      *reinterpret_cast<uint4*>(Wt + c * ldwt + r) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// e4m3 W codes [V, d] with row scales -> bf16 Wt [d, ldwt], vectorized as
// k_transpose_w_bf16 (8 codes per 8-byte load; d a multiple of 16). Each
// element is decoded exactly, multiplied by its row's scale in float32 and
// rounded to bf16 to nearest even, as the element-wise kernel does.
__global__ void __launch_bounds__(256) k_transpose_w_e4m3(const uint8_t* __restrict__ W,
                                                          const float* __restrict__ w_scale,
                                                          int64_t V, int64_t d,
                                                          __nv_bfloat16* __restrict__ Wt,
                                                          int64_t ldwt) {
  __shared__ float tile[kTT][kTT + 1];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTT;
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kTT;
  const int i = threadIdx.x >> 3, j = threadIdx.x & 7;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int rr = i + 32 * p;
    const int64_t r = r0 + rr, c = c0 + 8 * j;
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (r < V && c < d) {
      const uint2 q = *reinterpret_cast<const uint2*>(W + r * d + c);
      const float sc = w_scale[r];
      const uint32_t b[2] = {q.x, q.y};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        __nv_fp8_e4m3 v;
        v.__x = static_cast<uint8_t>((b[k >> 2] >> (8 * (k & 3))) & 0xFFu);
        f[k] = static_cast<float>(v) * sc;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) tile[rr][8 * j + k] = f[k];
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int cc = i + 32 * p;
    const int64_t c = c0 + cc, r = r0 + 8 * j;
    if (c < d && r < ldwt) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 h =
            __floats2bfloat162_rn(tile[8 * j + 2 * k][cc], tile[8 * j + 2 * k + 1][cc]);
        w[k] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(Wt + c * ldwt + r) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ----------------------------------------------------- compacted H^T
// Ht[c][r] = bf16(H[src(r)][c]) for compacted rows r in [0, nblk_max * 128):
// the row of block blk[r / 128] at offset r % 128, or 0 past the valid blocks
// or past N (those rows of dZ are 0, and 0 * garbage could be NaN).
template <int ELT>
__global__ void k_transpose_h_compact(const void* __restrict__ H,
                                      const float* __restrict__ h_scale, int64_t N, int64_t d,
                                      const int* __restrict__ blk, const int* nblk_dev,
                                      __nv_bfloat16* __restrict__ Ht, int64_t ldht) {
  __shared__ float tile[32][33];
  const int nb = *nblk_dev;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32;  // compacted rows
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * 32;  // hidden columns
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    const int64_t jb = r / kBM;
    float v = 0.f;
    if (jb < nb && c < d) {
      const int64_t src = static_cast<int64_t>(blk[jb]) * kBM + (r - jb * kBM);
      if (src < N) v = load_elt<ELT>(H, h_scale, src, src * d + c);
    }
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (c < d) Ht[c * ldht + r] = __float2bfloat16_rn(tile[threadIdx.x][i]);
  }
}

// ------------------------------------------------------ e4m3 quantization
// One warp per row, 16 consecutive elements per lane step (cols % 16 == 0,
// 16-byte aligned rows). amax = max |x| over the row; scale = amax / 448 and
// inv = 448 / amax with correctly rounded divisions (1 and 1 for a row of
// zeros); q = e4m3(x * inv), round to nearest even, saturated to +-448. The
// row is read twice; the second pass mostly hits L1/L2.
constexpr int kQuantRowsPerCta = 8;

template <bool F32>
__device__ __forceinline__ void load16(const void* x, int64_t e, float (&v)[16]) {
  if constexpr (F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + e);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 f = p[k];
      v[4 * k] = f.x;
      v[4 * k + 1] = f.y;
      v[4 * k + 2] = f.z;
      v[4 * k + 3] = f.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + e);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 u = p[k];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * k + 2 * j] = __uint_as_float(w[j] << 16);
        v[8 * k + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
}

template <bool F32>
__global__ void k_quantize_e4m3_rows(const void* __restrict__ x, int64_t rows, int64_t cols,
                                     uint8_t* __restrict__ q, float* __restrict__ scale) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kQuantRowsPerCta + warp;
  if (row >= rows) return;
  const int64_t ng = cols / 16;
  const int64_t base = row * cols;
  float amax = 0.f;
  for (int64_t gi = lane; gi < ng; gi += 32) {
    float v[16];
    load16<F32>(x, base + gi * 16, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const bool nz = amax > 0.f;
  const float inv = nz ? __fdiv_rn(448.f, amax) : 1.f;
  if (lane == 0) scale[row] = nz ? __fdiv_rn(amax, 448.f) : 1.f;
  for (int64_t gi = lane; gi < ng; gi += 32) {
    float v[16];
    load16<F32>(x, base + gi * 16, v);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t b = __nv_cvt_float_to_fp8(__fmul_rn(v[j], inv), __NV_SATFINITE, __NV_E4M3);
      w[j >> 2] |= (b & 0xFFu) << (8 * (j & 3));
    }
    *reinterpret_cast<uint4*>(q + base + gi * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------ zero rows
// Zero the output rows of every 128-row block that holds no valid token.
__global__ void k_zero_invalid_rows(const int* __restrict__ inv, int64_t N, int64_t row_bytes,
                                    uint8_t* __restrict__ out) {
  const int k = blockIdx.x;
  if (inv[k] >= 0) return;
  const int64_t r0 = static_cast<int64_t>(k) * kBM;
  const int64_t r1 = min(N, r0 + kBM);
  const int64_t n16 = (r1 - r0) * row_bytes / 16;
  uint4* p = reinterpret_cast<uint4*>(out + r0 * row_bytes);
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) p[i] = make_uint4(0, 0, 0, 0);
}

}  // namespace

cudaError_t launch_advantages(const float* rewards, int B, int G, float eps, int unbiased,
                              float* adv, cudaStream_t s) {
  const int groups = B / G;
  const int threads = 128;
  const int blocks = (groups * 32 + threads - 1) / threads;
  k_advantages<<<blocks, threads, 0, s>>>(rewards, B, G, eps, unbiased, adv);
  return cudaGetLastError();
}

cudaError_t launch_convert_bf16(const float* src, __nv_bfloat16* dst, int64_t n,
                                cudaStream_t s) {
  const int64_t vec = (n + 3) / 4;
  const int blocks = static_cast<int>(std::min<int64_t>((vec + 255) / 256, 8192));
  k_convert_bf16<<<blocks, 256, 0, s>>>(src, dst, n);
  return cudaGetLastError();
}

cudaError_t launch_seq_count(const uint8_t* mask, const int32_t* ids, int B, int T, int64_t V,
                             int* cnt, uint32_t* err, cudaStream_t s) {
  k_seq_count<<<B, 256, 0, s>>>(mask, ids, T, V, cnt, err);
  return cudaGetLastError();
}

cudaError_t launch_block_plan(const uint8_t* mask, int64_t N, int nblk, int* blk, int* inv,
                              int* nblk_dev, cudaStream_t s) {
  k_block_plan<<<1, 1024, 0, s>>>(mask, N, nblk, blk, inv, nblk_dev);
  return cudaGetLastError();
}

cudaError_t launch_fwd_finish(const int* inv, const uint8_t* mask, const int* cnt,
                              const float* adv, const float* zy, const float2* part,
                              int nblk_max, int n_vs, int64_t N, int B, int T, int token_level,
                              int ref_given, int kl_mode, float* logp_pol, float* logp_ref,
                              float* lse_pol, double* partials, int grid, cudaStream_t s) {
  k_fwd_finish<<<grid, 256, 0, s>>>(inv, mask, cnt, adv, zy, part, nblk_max, n_vs, N, B, T,
                                    token_level, ref_given, kl_mode, logp_pol, logp_ref, lse_pol,
                                    partials);
  return cudaGetLastError();
}

cudaError_t launch_fwd_reduce(const double* partials, int nparts, const int* cnt, int B,
                              float beta, int token_level, float* loss, float* kl_mean,
                              cudaStream_t s) {
  k_fwd_reduce<<<1, 32, 0, s>>>(partials, nparts, cnt, B, beta, token_level, loss, kl_mean);
  return cudaGetLastError();
}

cudaError_t launch_bwd_coef(const uint8_t* mask, const int* cnt, const float* adv,
                            const float* logp_pol, const float* logp_ref, int64_t N, int B,
                            int T, float beta, float grad, int token_level, int kl_mode,
                            float* coef, cudaStream_t s) {
  const int blocks = static_cast<int>(std::min<int64_t>((N + 255) / 256, 4096));
  k_bwd_coef<<<blocks, 256, 0, s>>>(mask, cnt, adv, logp_pol, logp_ref, N, B, T, beta, grad,
                                    token_level, kl_mode, coef);
  return cudaGetLastError();
}

cudaError_t launch_transpose_w(const void* W, int w_type, const float* w_scale, int64_t V,
                               int64_t d, __nv_bfloat16* Wt, int64_t ldwt, cudaStream_t s) {
  if (w_type == ELT_BF16 && d % 8 == 0 && ldwt % 8 == 0 &&
      (reinterpret_cast<uintptr_t>(W) & 15) == 0 && (reinterpret_cast<uintptr_t>(Wt) & 15) == 0) {
    // every column of Wt up to ldwt is written (zeros past V)
    dim3 grid(static_cast<unsigned>((ldwt + kTT - 1) / kTT),
              static_cast<unsigned>((d + kTT - 1) / kTT));
    k_transpose_w_bf16<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W), V, d, Wt,
                                            ldwt);
    return cudaGetLastError();
  }
  if (w_type == ELT_E4M3 && d % 8 == 0 && ldwt % 8 == 0 &&
      (reinterpret_cast<uintptr_t>(W) & 7) == 0 && (reinterpret_cast<uintptr_t>(Wt) & 15) == 0) {
    dim3 grid(static_cast<unsigned>((ldwt + kTT - 1) / kTT),
              static_cast<unsigned>((d + kTT - 1) / kTT));
    k_transpose_w_e4m3<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(W), w_scale, V, d, Wt,
                                            ldwt);
    return cudaGetLastError();
  }
  dim3 grid(static_cast<unsigned>((V + 31) / 32), static_cast<unsigned>((d + 31) / 32));
  dim3 block(32, 8);
  if (w_type == ELT_F32)
    k_transpose_w<ELT_F32><<<grid, block, 0, s>>>(W, w_scale, V, d, Wt, ldwt);
  else if (w_type == ELT_E4M3)
    k_transpose_w<ELT_E4M3><<<grid, block, 0, s>>>(W, w_scale, V, d, Wt, ldwt);
  else
    k_transpose_w<ELT_BF16><<<grid, block, 0, s>>>(W, w_scale, V, d, Wt, ldwt);
  return cudaGetLastError();
}

// bf16 H -> compacted Ht, vectorized as k_transpose_w_bf16: compacted row r
// of the tile comes from row blk[r / 128] * 128 + r % 128 of H, or is 0 past
// the valid blocks or past N.
__global__ void __launch_bounds__(256) k_transpose_h_bf16(const __nv_bfloat16* __restrict__ H,
                                                          int64_t N, int64_t d,
                                                          const int* __restrict__ blk,
                                                          const int* nblk_dev,
                                                          __nv_bfloat16* __restrict__ Ht,
                                                          int64_t ldht) {
  __shared__ float tile[kTT][kTT + 1];
  const int nb = *nblk_dev;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTT;  // compacted rows
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kTT;  // hidden columns
  const int i = threadIdx.x >> 3, j = threadIdx.x & 7;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int rr = i + 32 * p;
    const int64_t r = r0 + rr, c = c0 + 8 * j;
    const int64_t jb = r / kBM;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (jb < nb && c < d) {
      const int64_t src = static_cast<int64_t>(blk[jb]) * kBM + (r - jb * kBM);
      if (src < N) v = *reinterpret_cast<const uint4*>(H + src * d + c);
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      tile[rr][8 * j + 2 * k] = __uint_as_float(w[k] << 16);
      tile[rr][8 * j + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int cc = i + 32 * p;
    const int64_t c = c0 + cc, r = r0 + 8 * j;
    if (c < d && r < ldht) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = __float_as_uint(tile[8 * j + 2 * k][cc]) >> 16;
        const uint32_t hi = __float_as_uint(tile[8 * j + 2 * k + 1][cc]) & 0xFFFF0000u;
        w[k] = lo | hi;
      }
      *reinterpret_cast<uint4*>(Ht + c * ldht + r) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

cudaError_t launch_transpose_h_compact(const void* H, int h_type, const float* h_scale,
                                       int64_t N, int64_t d, const int* blk, const int* nblk_dev,
                                       int nblk_max, __nv_bfloat16* Ht, int64_t ldht,
                                       cudaStream_t s) {
  if (h_type == ELT_BF16 && d % 8 == 0 && ldht % 8 == 0 &&
      (reinterpret_cast<uintptr_t>(H) & 15) == 0 && (reinterpret_cast<uintptr_t>(Ht) & 15) == 0) {
    dim3 grid(static_cast<unsigned>((static_cast<int64_t>(nblk_max) * kBM + kTT - 1) / kTT),
              static_cast<unsigned>((d + kTT - 1) / kTT));
    k_transpose_h_bf16<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(H), N, d, blk,
                                            nblk_dev, Ht, ldht);
    return cudaGetLastError();
  }
  dim3 grid(static_cast<unsigned>(nblk_max * (kBM / 32)), static_cast<unsigned>((d + 31) / 32));
  dim3 block(32, 8);
  if (h_type == ELT_E4M3)
    k_transpose_h_compact<ELT_E4M3>
        <<<grid, block, 0, s>>>(H, h_scale, N, d, blk, nblk_dev, Ht, ldht);
  else
    k_transpose_h_compact<ELT_BF16>
        <<<grid, block, 0, s>>>(H, h_scale, N, d, blk, nblk_dev, Ht, ldht);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3_rows(const void* x, int x_f32, int64_t rows, int64_t cols,
                                      uint8_t* q, float* scale, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((rows + kQuantRowsPerCta - 1) / kQuantRowsPerCta);
  if (x_f32)
    k_quantize_e4m3_rows<true><<<grid, 32 * kQuantRowsPerCta, 0, s>>>(x, rows, cols, q, scale);
  else
    k_quantize_e4m3_rows<false><<<grid, 32 * kQuantRowsPerCta, 0, s>>>(x, rows, cols, q, scale);
  return cudaGetLastError();
}

cudaError_t launch_zero_invalid_rows(const int* inv, int64_t N, int64_t d, void* out,
                                     int out_f32, cudaStream_t s) {
  const int nblk = static_cast<int>((N + kBM - 1) / kBM);
  k_zero_invalid_rows<<<nblk, 256, 0, s>>>(inv, N, d * (out_f32 ? 4 : 2),
                                           static_cast<uint8_t*>(out));
  return cudaGetLastError();
}

}  // namespace grpo

// ge_norm.cu -- the normalisation pass of MatMul + bias + residual +
// RMSNorm / LayerNorm (ops-nn MatMul fusion (codearts), "ops-nn's MatMul
// fusion strategy", second level: the norm reduces across the channel
// dimension, so it cannot be applied element by element in the GEMM's
// epilogue). The GEMM epilogue has already written h = A.B + bias +
// residual as H:
//
//   RMSNorm:   y = h * rsqrt(mean(h^2) + eps) * gamma
//   LayerNorm: y = (h - mu) * rsqrt(mean((h - mu)^2) + eps) * gamma + beta
//
// Tensor-core path: the GEMM epilogue also took each token's statistics
// (per tile); norm_finalize_kernel merges them into (mean, rstd) per token
// and norm_apply_kernel streams H -> Y elementwise (one read of H, one
// write of Y: HBM-bound, no reductions on the way).
// GEMV path and unfused flow: norm_kernel takes the statistics itself, one
// block per token, the row in registers, two exact passes (mean, then
// squared deviations) rather than a sum of squares minus a squared mean.
#include "ge_elem.cuh"
#include "ge_internal.h"
#include "ge_ptx.cuh"

namespace ge {
namespace {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// No "memory" clobber: the compiler may then issue the read-only gamma /
// beta loads of later groups before these stores. H is read through the
// volatile ld_stream, which stays ordered with these volatile stores, so Y
// may still be H.
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w));
}

// Y's 8 values of group g from H's values v, with gamma / beta.
__device__ __forceinline__ uint4 norm8(const uint4& v, const uint4& gm, const uint4& bt, float mu, float rstd,
                                       bool layer, bool bf16) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const uint32_t gw[4] = {gm.x, gm.y, gm.z, gm.w};
  const uint32_t bw[4] = {bt.x, bt.y, bt.z, bt.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = to_f32x2(bf16, w[k]);
    const float2 gg = to_f32x2(bf16, gw[k]);
    const float2 bb = layer ? to_f32x2(bf16, bw[k]) : make_float2(0.0f, 0.0f);
    o[k] = pack2(bf16, fmaf((x.x - mu) * rstd, gg.x, bb.x), fmaf((x.y - mu) * rstd, gg.y, bb.y));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

// Sum over the eight 16-bit values of `v` of f(x).
template <class F>
__device__ __forceinline__ float sum8(const uint4& v, bool bf16, F f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = to_f32x2(bf16, w[i]);
    s += f(x.x) + f(x.y);
  }
  return s;
}

// Norm of whole rows of H when no statistics were taken upstream (the GEMV
// path, N <= 16 tokens, and the unfused flow): one 256-thread block per row.
// Thread t keeps the row's 16-byte groups t, t + 256, ... (up to BLOCK_CACHE
// of them: 8192 features) in registers; two block reductions give the mean
// and the variance exactly (two passes over registers); a third pass writes
// Y. Longer rows re-read their remainder (from L2) in each pass.
constexpr int BLOCK_CACHE = 4;

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5;
  __syncthreads();  // red may still be read by the previous reduction
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) t += red[i];  // fixed order: the same sum in every thread
  return t;
}

__global__ void __launch_bounds__(256) norm_kernel(const NormArgs p) {
  __shared__ float red[8];
  const bool bf16 = p.bf16 != 0;
  const bool layer = p.layer != 0;
  const long long G = p.C >> 3;  // whole 16-byte groups per row
  const float inv_c = 1.0f / static_cast<float>(p.C);
  const int t = threadIdx.x;
  for (long long r = blockIdx.x; r < p.R; r += gridDim.x) {
    const unsigned short* h = p.H + r * p.ld;
    unsigned short* y = p.Y + r * p.ld;
    uint4 cache[BLOCK_CACHE];
#pragma unroll
    for (int i = 0; i < BLOCK_CACHE; ++i) {
      const long long g = t + 256LL * i;
      cache[i] = g < G ? ld_stream(h + 8 * g) : make_uint4(0, 0, 0, 0);
    }
    // the C % 8 features past the last whole group: one per thread
    const long long tail_c = 8 * G + t;
    const bool has_tail = tail_c < p.C;
    const float tail = has_tail ? to_f32(bf16, h[tail_c]) : 0.0f;
    auto for_groups = [&](auto&& fn) {
#pragma unroll
      for (int i = 0; i < BLOCK_CACHE; ++i) {
        const long long g = t + 256LL * i;
        if (g < G) fn(cache[i], g);
      }
      for (long long g = t + 256LL * BLOCK_CACHE; g < G; g += 256) fn(ld_stream(h + 8 * g), g);
    };
    float mu = 0.0f;
    if (layer) {
      float s = tail;
      for_groups([&](const uint4& v, long long) { s += sum8(v, bf16, [](float x) { return x; }); });
      mu = block_sum(s, red) * inv_c;
    }
    float ss = has_tail ? (tail - mu) * (tail - mu) : 0.0f;
    for_groups([&](const uint4& v, long long) {
      ss += sum8(v, bf16, [mu](float x) { return (x - mu) * (x - mu); });
    });
    const float rstd = rsqrtf(block_sum(ss, red) * inv_c + p.eps);
    for_groups([&](const uint4& v, long long g) {
      const uint4 gm = __ldg(reinterpret_cast<const uint4*>(p.gamma) + g);
      const uint4 bt = layer ? __ldg(reinterpret_cast<const uint4*>(p.beta) + g) : make_uint4(0, 0, 0, 0);
      st_stream(y + 8 * g, norm8(v, gm, bt, mu, rstd, layer, bf16));
    });
    if (has_tail) {
      const float bb = layer ? to_f32(bf16, p.beta[tail_c]) : 0.0f;
      y[tail_c] = from_f32(bf16, fmaf((tail - mu) * rstd, to_f32(bf16, p.gamma[tail_c]), bb));
    }
  }
}

// Features of tile t's 32-feature slabs c with c % halves == half: the tile
// holds v = min(tile_w, C - t*tile_w) features, v / 32 whole slabs and one
// slab of v % 32.
__device__ __forceinline__ float half_count(long long C, int tile_w, int t, int half, int halves) {
  const long long left = C - static_cast<long long>(t) * tile_w;
  const int v = left < tile_w ? static_cast<int>(left) : tile_w;
  const int full = v >> 5;
  const int whole = (full + halves - 1 - half) / halves;  // whole slabs c < full with c % halves == half
  return static_cast<float>(32 * whole + (full % halves == half ? (v & 31) : 0));
}

// Chan's merge of two (count, mean, sum of squared deviations) summaries.
__device__ __forceinline__ void chan_merge(float& n, float& mean, float& m2, float nb, float mb, float m2b) {
  const float nn = n + nb;
  if (nn == 0.0f) return;
  const float delta = mb - mean;
  const float w = __fdividef(nb, nn);  // counts are integers below 2^24: a fast divide is exact enough
  mean = fmaf(delta, w, mean);
  m2 = m2 + m2b + delta * delta * (n * w);
  n = nn;
}

// Statistics taken by the GEMM epilogue: one warp per row. Lane l merges
// partials l, l + 32, ... in order, then a fixed shuffle tree merges the
// lanes (lower lane on the left at every level), so the result does not
// depend on timing. Writes (mean, rstd) of the row.
__global__ void __launch_bounds__(256) norm_finalize_kernel(const NormArgs p) {
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  const long long nwarps = static_cast<long long>(gridDim.x) * wpb;
  const int np = p.halves * p.ntiles;
  for (long long r = blockIdx.x * wpb + (threadIdx.x >> 5); r < p.R; r += nwarps) {
    float n = 0.0f, mean = 0.0f, m2 = 0.0f;
    for (int k = lane; k < np; k += 32) {
      const float2 s = __ldcg(p.partials + static_cast<long long>(k) * p.R + r);
      float nb;
      if (p.halves == 1) {  // one partial per tile: its features
        const long long left = p.C - static_cast<long long>(k) * p.tile_w;
        nb = static_cast<float>(left < p.tile_w ? left : p.tile_w);
      } else {
        nb = half_count(p.C, p.tile_w, k / p.halves, k % p.halves, p.halves);
      }
      chan_merge(n, mean, m2, nb, s.x, s.y);
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float on = __shfl_xor_sync(0xffffffffu, n, off);
      const float om = __shfl_xor_sync(0xffffffffu, mean, off);
      const float o2 = __shfl_xor_sync(0xffffffffu, m2, off);
      if (lane & off) {  // this lane holds the right operand: merge into the partner's (left) copy
        float ln = on, lm = om, l2 = o2;
        chan_merge(ln, lm, l2, n, mean, m2);
        n = ln;
        mean = lm;
        m2 = l2;
      } else {
        chan_merge(n, mean, m2, on, om, o2);
      }
    }
    if (lane == 0) {
      const float inv_c = 1.0f / static_cast<float>(p.C);
      // LayerNorm: variance about the mean; RMSNorm: mean square (M2 + C mean^2) / C
      const float ms = p.layer ? m2 * inv_c : fmaf(mean, mean, m2 * inv_c);
      p.rowstats[r] = make_float2(p.layer ? mean : 0.0f, rsqrtf(ms + p.eps));
    }
  }
}

// y = (h - mean) * rstd * gamma + beta for every element: units of 8
// features, two per thread 256 apart inside the block's chunk, both loads
// issued before the stores (the layout of the other elementwise passes,
// which run at copy speed).
template <int F>
__global__ void __launch_bounds__(256) norm_apply_kernel(const NormArgs p) {
  const bool bf16 = p.bf16 != 0;
  const bool layer = p.layer != 0;
  const long long G = p.C >> 3;
  const long long total = p.R * G;
  constexpr int U = 2;
  const long long step = (F & F_BIG) ? static_cast<long long>(gridDim.x) * 256 * U : total;
  for (long long i0 = blockIdx.x * (256LL * U) + threadIdx.x; i0 < total; i0 += step) {
    uint4 v[U];
    long long rr[U], gg[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = i0 + u * 256;
      rr[u] = gg[u] = 0;
      v[u] = make_uint4(0, 0, 0, 0);
      if (i < total) {
        split_index<F>(i, G, rr[u], gg[u]);
        v[u] = ld_stream(p.H + rr[u] * p.ld + 8 * gg[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i0 + u * 256 >= total) continue;
      const float2 st = __ldg(p.rowstats + rr[u]);
      const uint4 gm = __ldg(reinterpret_cast<const uint4*>(p.gamma) + gg[u]);
      const uint4 bt = layer ? __ldg(reinterpret_cast<const uint4*>(p.beta) + gg[u]) : make_uint4(0, 0, 0, 0);
      st_stream(p.Y + rr[u] * p.ld + 8 * gg[u], norm8(v[u], gm, bt, st.x, st.y, layer, bf16));
    }
  }
}

// The C % 8 features past the last whole group of every row, one thread
// each (launched only when C is not a multiple of 8).
__global__ void __launch_bounds__(256) norm_apply_tail_kernel(const NormArgs p) {
  const bool bf16 = p.bf16 != 0;
  const bool layer = p.layer != 0;
  const long long c0 = p.C & ~7LL;
  const long long tail = p.C - c0;
  const long long stride = static_cast<long long>(gridDim.x) * 256;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < p.R * tail; i += stride) {
    const long long r = i / tail;
    const long long c = c0 + (i - r * tail);
    const float2 st = p.rowstats[r];
    const float x = to_f32(bf16, p.H[r * p.ld + c]);
    const float b = layer ? to_f32(bf16, p.beta[c]) : 0.0f;
    p.Y[r * p.ld + c] = from_f32(bf16, fmaf((x - st.x) * st.y, to_f32(bf16, p.gamma[c]), b));
  }
}

// H += residual in place; units of 8 contiguous elements, two per thread
// 256 apart inside the block's chunk, all loads issued before the stores.
template <int F>
__global__ void __launch_bounds__(256) residual_add_kernel(unsigned short* D, long long R, long long C,
                                                           long long ld, const unsigned short* res,
                                                           int bf16_flag) {
  const bool bf16 = bf16_flag != 0;
  const long long per_row = (C + 7) / 8;
  const long long total = R * per_row;
  constexpr int U = 2;
  const long long step = (F & F_BIG) ? static_cast<long long>(gridDim.x) * 256 * U : total;
  for (long long i0 = blockIdx.x * (256LL * U) + threadIdx.x; i0 < total; i0 += step) {
    uint4 va[U], vb[U];
    long long off[U], cc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = i0 + u * 256;
      cc[u] = C;
      off[u] = 0;
      va[u] = vb[u] = make_uint4(0, 0, 0, 0);
      if (i < total) {
        long long r, k;
        split_index<F>(i, per_row, r, k);
        cc[u] = k * 8;
        off[u] = r * ld + cc[u];
        va[u] = load_unit<F>(D + off[u], cc[u], C);
        vb[u] = load_unit<F>(res + off[u], cc[u], C);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (cc[u] >= C) continue;
      const uint32_t aw[4] = {va[u].x, va[u].y, va[u].z, va[u].w};
      const uint32_t bw[4] = {vb[u].x, vb[u].y, vb[u].z, vb[u].w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = to_f32x2(bf16, aw[k]);
        const float2 z = to_f32x2(bf16, bw[k]);
        o[k] = pack2(bf16, x.x + z.x, x.y + z.y);
      }
      store_unit<F>(D + off[u], make_uint4(o[0], o[1], o[2], o[3]), cc[u], C);
    }
  }
}

}  // namespace

cudaError_t launch_norm(const NormArgs& a, int num_sms, cudaStream_t s) {
  if (a.R == 0 || a.C == 0) return cudaSuccess;
  if (a.partials) {
    long long fb = (a.R + 7) / 8;  // one row per warp
    if (fb > static_cast<long long>(num_sms) * 16) fb = static_cast<long long>(num_sms) * 16;
    norm_finalize_kernel<<<static_cast<unsigned>(fb), 256, 0, s>>>(a);
    const long long units = a.R * (a.C >> 3);
    if (units > 0) {
      long long blocks = (units + 511) / 512;  // two units per thread
      const bool big = blocks > 65535LL * 8 || units > (1LL << 32);
      if (blocks > 65535LL * 8) blocks = 65535LL * 8;
      if (big)
        norm_apply_kernel<F_BIG><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
      else
        norm_apply_kernel<0><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    }
    if (a.C & 7) {
      long long tb = (a.R * (a.C & 7) + 255) / 256;
      if (tb > 65535LL * 8) tb = 65535LL * 8;
      norm_apply_tail_kernel<<<static_cast<unsigned>(tb), 256, 0, s>>>(a);
    }
    return cudaGetLastError();
  }
  long long blocks = a.R;  // one row per block
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  norm_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_residual_add(__half* D, long long R, long long C, long long ld,
                                const unsigned short* res, int bf16, cudaStream_t s) {
  if (R == 0 || C == 0) return cudaSuccess;
  const long long units = R * ((C + 7) / 8);
  long long blocks = (units + 511) / 512;  // two units per thread
  int f = C % 8 != 0 ? F_RAGGED : 0;
  if (blocks > 65535LL * 8 || units > (1LL << 32)) f |= F_BIG;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  unsigned short* d = reinterpret_cast<unsigned short*>(D);
  const unsigned g = static_cast<unsigned>(blocks);
  switch (f) {
    case 0: residual_add_kernel<0><<<g, 256, 0, s>>>(d, R, C, ld, res, bf16); break;
    case F_RAGGED: residual_add_kernel<F_RAGGED><<<g, 256, 0, s>>>(d, R, C, ld, res, bf16); break;
    case F_BIG: residual_add_kernel<F_BIG><<<g, 256, 0, s>>>(d, R, C, ld, res, bf16); break;
    default: residual_add_kernel<F_RAGGED | F_BIG><<<g, 256, 0, s>>>(d, R, C, ld, res, bf16);
  }
  return cudaGetLastError();
}

}  // namespace ge

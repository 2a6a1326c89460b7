// ge_elem.cuh -- device helpers shared by the HBM-bound elementwise passes
// (the unfused baseline's bias add and activation, the residual add): the
// launch-time specialisation flags and the loads and stores of one unit of
// 8 contiguous 16-bit elements, partial at a ragged row end.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace ge {

// Launch-time specialisations of the elementwise kernels. Each is decided
// once per launch on the host, so the common case carries no code for the
// others.
constexpr int F_RAGGED = 1;  // C % 8 != 0: a row's last unit is partial
constexpr int F_BIG = 2;     // 64-bit index arithmetic and a grid-stride loop
constexpr int F_MASK = 4;    // RELU_AUX_BIAS: write the mask words
constexpr int F_ZAUX = 8;    // GELU_AUX_BIAS: keep the pre-activation z

// The ragged end of a row (n < 8 columns left) goes through the same
// arithmetic as a full unit: its elements are gathered into a zero-padded
// 16-byte value (zero activates to zero and sets no mask bit) and only the
// n real ones are written back.
__device__ __forceinline__ uint4 load_partial(const unsigned short* p, int n) {
  unsigned long long lo = 0, hi = 0;
  for (int k = 0; k < n; ++k) {
    const unsigned long long e = p[k];
    if (k < 4)
      lo |= e << (16 * k);
    else
      hi |= e << (16 * (k - 4));
  }
  return make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32), static_cast<uint32_t>(hi),
                    static_cast<uint32_t>(hi >> 32));
}

__device__ __forceinline__ void store_partial(unsigned short* p, const uint4& v, int n) {
  const unsigned long long lo = v.x | (static_cast<unsigned long long>(v.y) << 32);
  const unsigned long long hi = v.z | (static_cast<unsigned long long>(v.w) << 32);
  for (int k = 0; k < n; ++k)
    p[k] = static_cast<unsigned short>(k < 4 ? lo >> (16 * k) : hi >> (16 * (k - 4)));
}

// Unit u of a row-major [R][per_row units] index space -> (row, unit in row).
template <int F>
__device__ __forceinline__ void split_index(long long q, long long per_row, long long& r, long long& k) {
  if constexpr (F & F_BIG) {
    r = q / per_row;
  } else {
    r = static_cast<uint32_t>(q) / static_cast<uint32_t>(per_row);
  }
  k = q - r * per_row;
}

template <int F>
__device__ __forceinline__ uint4 load_unit(const unsigned short* p, long long c0, long long C) {
  if (c0 + 8 <= C || !(F & F_RAGGED)) return *reinterpret_cast<const uint4*>(p);
  return load_partial(p, static_cast<int>(C - c0));
}

template <int F>
__device__ __forceinline__ void store_unit(unsigned short* p, const uint4& v, long long c0, long long C) {
  if (c0 + 8 <= C || !(F & F_RAGGED))
    *reinterpret_cast<uint4*>(p) = v;
  else
    store_partial(p, v, static_cast<int>(C - c0));
}

}  // namespace ge

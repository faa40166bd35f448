// Top-k routing of one token by one warp, shared by the routing kernels of the
// paged fused MoE layer (the standard top-k MoE router: softmax over the
// experts' logits, the k largest kept, weights renormalised over them).
#pragma once

#include <cfloat>
#include <cstdint>

#include "device.cuh"

namespace rimuru {
namespace dev {

// Order-preserving 32-bit key of a float: a > b as floats iff key(a) > key(b).
// -0 is folded onto +0 first so the two compare equal, as IEEE says.
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Routing of one token by one warp.  Lane l holds experts l, l + 32, ...
// (EPL per lane) as keys; each of the k rounds takes the largest untaken key
// of the warp with one redux.max and, among lanes holding it, the lowest
// expert index with one redux.min.  Key 0 marks lanes past E (valid keys are
// >= key(-inf) > 0).  Lane j < k receives slot j: its expert and weight.
template <int EPL>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k,
                                            int renorm, int lane, int* err, int& my_id,
                                            float& my_w) {
  uint32_t key[EPL];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0u;
    if (e < E) {
      float x = row[e];
      if (!isfinite(x)) {
        bad = true;
        x = -INFINITY;  // invalid input: rank it last, keep ids valid
      }
      key[i] = order_key(x);
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, RIMURU_DEV_NONFINITE);
  // k selection rounds; lane j keeps the logit and expert of slot j, and the
  // exponentials are taken afterwards, one per lane, instead of once per round.
  uint32_t taken = 0, my_key = 0u;
  my_id = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u, bi = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (!((taken >> i) & 1u) && key[i] > bk) {  // strict: lowest index among equals
        bk = key[i];
        bi = static_cast<uint32_t>(lane + 32 * i);
      }
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t win = __reduce_min_sync(0xffffffffu, bk == m ? bi : 0xffffffffu);
    if (static_cast<int>(win & 31u) == lane) taken |= 1u << (win >> 5);
    if (lane == j) {
      my_id = static_cast<int>(win);
      my_key = m;
    }
  }
  // largest logit of the token: slot 0's (0 if it is -inf, i.e. no finite logit)
  const float top = key_value(__shfl_sync(0xffffffffu, my_key, 0));
  const float mx = (top == -INFINITY) ? 0.f : top;
  const float my_p = lane < k ? expf(key_value(my_key) - mx) : 0.f;
  float psum = my_p;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
  float denom = psum;
  if (!renorm) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (key[i] != 0u) s += expf(key_value(key[i]) - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    denom = s;
  }
  my_w = my_p / denom;
}

}  // namespace dev
}  // namespace rimuru

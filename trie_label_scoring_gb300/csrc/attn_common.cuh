// Device helpers shared by the two doc-attention kernels (mma.sync path in
// attention.cu, tcgen05 path in attention_tc.cu): RoPE angles, two-term bf16
// splits and the row -> (document, node) mapping.
#pragma once
#include <cmath>

#include "kernels.h"

namespace quail {

constexpr float kAttnLog2e = 1.4426950408889634f;

struct RopeTable {
  float2 w[64];  // inv_freq_j = theta^(-2j/128) as hi + lo floats
};

inline RopeTable make_rope_table(float theta) {
  RopeTable t;
  for (int j = 0; j < 64; ++j) {
    const double w = std::pow(static_cast<double>(theta), -2.0 * j / 128.0);
    const float hi = static_cast<float>(w);
    t.w[j] = make_float2(hi, static_cast<float>(w - static_cast<double>(hi)));
  }
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
}
// Two-term bf16 split of (x0, x1): hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  const float2 h = unpack_bf16(hi);
  lo = pack_bf16(x0 - h.x, x1 - h.y);
}

// cos/sin of pos * w, w given as hi + lo floats; exact product and a two-step
// reduction by 2*pi keep the angle accurate to ~1e-7 rad for pos < 2^24.
__device__ __forceinline__ void rope_cs(int pos, float2 w, float& c, float& s) {
  const float p = static_cast<float>(pos);
  const float a = p * w.x;
  const float b = fmaf(p, w.x, -a) + p * w.y;
  const float k = rintf(a * 0.15915494309189535f);
  float r = fmaf(-k, 6.28318548202514648f, a);  // 2*pi rounded to float
  r = fmaf(-k, -1.7484556000744487e-07f, r);    // 2*pi - float(2*pi)
  r += b;
  __sincosf(r, &s, &c);  // |r| <= pi + tiny: hardware sin/cos, absolute error ~4e-7
}

// 2^x with flush-to-zero (one MUFU op); used where x <= 8 and tiny results
// are negligible (softmax weights).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int row_doc(const RowMap& m, int slot) { return m.slot_doc ? m.slot_doc[slot] : slot; }
__device__ __forceinline__ int row_node(const RowMap& m, int slot, int e) {
  if (m.slot_base) {
    const int n = m.slot_rows[slot];
    return m.slot_base[slot] + (e < n ? e : n - 1);
  }
  return m.slot_node ? m.slot_node[slot] : slot * m.slot_stride + (m.row_nodes ? m.row_nodes[e] : e);
}
// True when every query row from e on is padding of its slot.
__device__ __forceinline__ bool rows_past_end(const RowMap& m, int slot, int e) {
  return m.slot_rows != nullptr && e >= m.slot_rows[slot];
}

}  // namespace quail

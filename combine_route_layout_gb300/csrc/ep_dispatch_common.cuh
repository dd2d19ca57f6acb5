// Device helpers shared by the dispatch kernels: the
// destination slot of a token on each rank, the per-row metadata a received
// row carries (MORI-EP User Guide, section 3, dispatch() return values), and
// the FP8 / FP4 block quantisers.
#pragma once

#include "ep_kernels.cuh"

namespace ep {
namespace {


// Slot of this token on rank `lane` (2D layout), or -1.
__device__ __forceinline__ int slot_on_lane_rank(const DispatchParams& p, int64_t g, int s, int t,
                                                 uint32_t m, int lane) {
  if (lane < p.R && ((m >> lane) & 1u)) {
    const int c = s * p.cpr + t / kChunk;
    const int local = __ldg(p.local8 + g * p.R + lane);
    if (!p.chunk_cnt) return __ldg(p.chunk_off + (int64_t)c * p.R + lane) + local;
    int off = 0;  // small batch: at most kSmallScanChunks - 1 earlier chunks
#pragma unroll 4
    for (int cc = 0; cc < c; ++cc) off += __ldg(p.chunk_cnt + (int64_t)cc * p.R + lane);
    return off + local;
  }
  return -1;
}

// Small batches: recv_num_token from the chunk counts (CTA 0, after the layout).
__device__ __forceinline__ void recv_from_counts(const DispatchParams& p) {
  if (!p.chunk_cnt || blockIdx.x != 0 || (int)threadIdx.x >= p.R) return;
  int n = 0;
  for (int cc = 0; cc < p.R * p.cpr; ++cc) n += __ldg(p.chunk_cnt + (int64_t)cc * p.R + threadIdx.x);
  p.recv_num_token[threadIdx.x] = n;
}

// Pool row (rank_base[owner] + row in the owner's region) of slot `lane`
// (standard MoE), or -1.
__device__ __forceinline__ int64_t row_on_lane_slot(const DispatchParams& p, int64_t g, int s,
                                                    int t, int lane) {
  if (lane >= p.k) return -1;
  const int e = __ldg(p.idx + g * p.k + lane);
  if (e < 0 || e >= p.E) return -1;
  const int l = __ldg(p.local16 + g * p.k + lane);
  if (l == 0xFFFF) return -1;
  const int c = s * p.cpr + t / kChunk;
  const int64_t row = (int64_t)__ldg(p.rank_base + e / p.E_r) + __ldg(p.expert_offset + e) +
                      __ldg(p.chunk_off + (int64_t)c * p.E + e) + l;
  if (row >= p.cap) return -1;  // capacity overflow is flagged by the layout kernel
  return row;
}

// Pass-through scale row of token g to receive row `row` (4-byte words when possible).
__device__ __forceinline__ void copy_scale_row(const DispatchParams& p, int64_t g, int64_t row,
                                               int lane) {
  if ((p.scale_row_bytes & 3) == 0) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.scales_in + g * p.scale_row_bytes);
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.out_scales + row * p.scale_row_bytes);
    for (int i = lane; i < (p.scale_row_bytes >> 2); i += 32) dst[i] = __ldg(src + i);
  } else {
    const uint8_t* src = p.scales_in + g * p.scale_row_bytes;
    uint8_t* dst = p.out_scales + row * p.scale_row_bytes;
    for (int i = lane; i < p.scale_row_bytes; i += 32) dst[i] = __ldg(src + i);
  }
}

// Per-destination metadata of the 2D layout (segment 0 of a token only).
__device__ void write_meta_2d(const DispatchParams& p, int64_t g, int s, int t, uint32_t m,
                              int my_slot, int lane) {
  if (lane < p.R) p.slot_map[g * p.R + lane] = my_slot;
  if (my_slot >= 0) p.src_pos[(int64_t)lane * p.cap + my_slot] = s * (p.R * p.Tmax) + t;
  const float wv = lane < p.k ? __ldg(p.w + g * p.k + lane) : 0.f;
  const int iv = lane < p.k ? __ldg(p.idx + g * p.k + lane) : 0;
  for (uint32_t mm = m; mm; mm &= mm - 1) {
    const int r = __ffs(mm) - 1;
    const int sl = __shfl_sync(kFull, my_slot, r);
    const int64_t row = (int64_t)r * p.cap + sl;
    if (lane < p.k) {
      p.out_w[row * p.k + lane] = wv;
      p.out_idx[row * p.k + lane] = iv;
    }
    if (p.scale_row_bytes > 0 && p.scales_in) copy_scale_row(p, g, row, lane);
  }
}

// Per-slot metadata of the standard-MoE layout (segment 0 of a token only).
__device__ void write_meta_std(const DispatchParams& p, int64_t g, int s, int t, int64_t my_row,
                               int lane) {
  if (lane < p.k) {
    p.row_map[g * p.k + lane] = (int32_t)my_row;
    if (my_row >= 0) p.src_pos[my_row] = s * (p.R * p.Tmax) + t;
  }
  if (p.scale_row_bytes > 0 && p.scales_in) {
    for (uint32_t mm = __ballot_sync(kFull, my_row >= 0); mm; mm &= mm - 1) {
      const int j = __ffs(mm) - 1;
      copy_scale_row(p, g, __shfl_sync(kFull, my_row, j), lane);
    }
  }
}

// ----------------------------------------------------------- block quantisers
// bf16 in. Lane covers 16 consecutive elements (two 16-byte loads) per
// 512-element step, so 8 lanes cover one 128-element block; the block's amax
// is reduced with three xor-shuffles inside that 8-lane group.

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float f[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

// x / scale rounded to nearest even, for |x| <= amax = scale * 448 (or * 6),
// from rcp = 1/scale correctly rounded: the product q0 = x * rcp is within
// two ulps of the quotient, the residual x - q0 * scale is exact in one
// fused multiply-add, and one more fused multiply-add with rcp rounds the
// corrected quotient (Markstein's correction step). The residual is exact
// while it does not underflow, which holds for every |x| >= 2^-103; with
// amax >= kRcpMinAmax any smaller x quotes below 2^-14, far under half the
// smallest nonzero code (2^-10 for E4M3, 0.25 for E2M1), so its code (a
// signed zero) does not depend on the last bits. Blocks with a smaller amax are scaled by 2^100 first (x and
// the scale, both exactly, so the quotient is unchanged). An all-zero block
// (scale 0) gets rcp = 0, which turns every quotient into a zero of x's
// sign, the code of x / 0 as the block quantiser defines it. The sign bit of
// x is put back for x = -0 (the residual step would make it +0). Four
// floating-point operations instead of a full division per element, with no
// branch; every (x, amax) pair of bf16 values is checked against the IEEE
// quotient's code on the GPU.
constexpr float kRcpMinAmax = 0x1p-80f;

__device__ __forceinline__ float quotient(float x, float scale, float rcp) {
  const float q0 = __fmul_rn(x, rcp);
  const float r = __fmaf_rn(-q0, scale, x);
  const float q = __fmaf_rn(r, rcp, q0);
  return __int_as_float(__float_as_int(q) | (__float_as_int(x) & 0x80000000));
}

// RCP: quotients from the reciprocal and residual (above); otherwise by IEEE
// division. Both give the same codes.
template <bool RCP>
__device__ __forceinline__ void quant16(const uint4& a, const uint4& b, uint4& q, float& scale) {
  float f[16];
  unpack16(a, b, f);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
  scale = __fdiv_rn(amax, 448.0f);
  // blocks below kRcpMinAmax: x and scale times 2^100 (exact, same quotient);
  // all-zero blocks: rcp = 0, every quotient a zero of x's sign
  uint32_t c[8];
  if (RCP) {
    const float k = amax < kRcpMinAmax ? 0x1p100f : 1.0f;
    const float sk = scale * k;
    const float rcp = amax == 0.f ? 0.0f : __frcp_rn(sk);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      c[i] = cvt_e4m3x2(quotient(f[2 * i] * k, sk, rcp), quotient(f[2 * i + 1] * k, sk, rcp));
  } else if (amax == 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = cvt_e4m3x2(f[2 * i], f[2 * i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      c[i] = cvt_e4m3x2(__fdiv_rn(f[2 * i], scale), __fdiv_rn(f[2 * i + 1], scale));
  }
  q.x = c[0] | (c[1] << 16);
  q.y = c[2] | (c[3] << 16);
  q.z = c[4] | (c[5] << 16);
  q.w = c[6] | (c[7] << 16);
}

// FP4 with a whole 32-element block per lane (32 consecutive elements, four
// 16-byte loads): the block's amax needs no shuffle, and each destination row
// takes one 16-byte store of codes and one 4-byte scale store per lane.
__device__ __forceinline__ void quant32_fp4(const uint4 v[4], uint4& q, float& scale) {
  const uint32_t w[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                          v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  scale = __fdiv_rn(amax, 6.0f);
  // as in quant16: tiny blocks scaled by 2^100, all-zero blocks rcp = 0
  const float k = amax < kRcpMinAmax ? 0x1p100f : 1.0f;
  const float sk = scale * k;
  const float rcp = amax == 0.f ? 0.0f : __frcp_rn(sk);
  uint32_t out[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = bf16_lo(w[4 * h + j]);
      f[2 * j + 1] = bf16_hi(w[4 * h + j]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = quotient(f[j] * k, sk, rcp);
    out[h] = cvt_e2m1x8(f);
  }
  q = make_uint4(out[0], out[1], out[2], out[3]);
}

}  // namespace
}  // namespace ep

// Dispatch payload movement (the second half of dispatch).
//
// MORI-EP User Guide, section 3, dispatch(): each received row carries the
// token's payload, its weights and indices, and its scales. "Choosing an EP
// API and backend" lists quantization as a dispatch feature and fixes the FP8
// format to OCP E4M3; here the block is 128 elements with one f32 scale,
// scale = amax / 448, codes = E4M3 round-to-nearest-even saturating of x/scale.
//
// Work is split into units of (token, column segment); each warp takes units
// in a grid-stride loop, so all warps stay busy whatever the routing skew
// (the unit count depends only on the source tokens). A unit loads its
// segment of the source row once (16-byte non-coherent loads, all issued
// before any dependent work) and writes it to every destination, so HBM sees
// one read per token and one write per (token, destination). Segment 0 also
// writes the per-row metadata. The destination slot is the chunk offset plus
// the token's rank inside its chunk, both produced by the layout kernel.
#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

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

// Packed row (global index r*pcap + row) of slot `lane` (standard MoE), or -1.
__device__ __forceinline__ int64_t row_on_lane_slot(const DispatchParams& p, int64_t g, int s,
                                                    int t, int lane) {
  if (lane >= p.k) return -1;
  const int e = __ldg(p.idx + g * p.k + lane);
  if (e < 0 || e >= p.E) return -1;
  const int l = __ldg(p.local16 + g * p.k + lane);
  if (l == 0xFFFF) return -1;
  const int c = s * p.cpr + t / kChunk;
  const int64_t row =
      (int64_t)__ldg(p.expert_offset + e) + __ldg(p.chunk_off + (int64_t)c * p.E + e) + l;
  if (row >= p.cap) return -1;  // capacity overflow is flagged by the layout kernel
  return (int64_t)(e / p.E_r) * p.cap + row;
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

// ------------------------------------------------------------------ copy mode
// Payload bits are moved unchanged: lane covers 16 bytes per 512-byte step.

template <bool STD>
__global__ void __launch_bounds__(256, 4) dispatch_copy_kernel(DispatchParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  bool waited = false;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < p.total_units;
       u += nwarps) {
    const int64_t g = u / p.segs_per_token;
    const int seg = (int)(u - g * p.segs_per_token);
    const int s = (int)(g / p.Tmax), t = (int)(g - (int64_t)s * p.Tmax);
    if (t >= p.ntok[s]) continue;

    const uint8_t* src = p.x + g * p.in_row_bytes;
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int i = 0; i < kCopyUnroll; ++i) {
      const int64_t off = ((int64_t)seg * kCopyUnroll + i) * 512 + lane * 16;
      if (off < p.in_row_bytes) v[i] = ld_nc_v4(src + off);
    }
    if (!waited) {  // the routing layout is complete and visible past this point
      pdl_wait();
      waited = true;
    }

    if (!STD) {
      const uint32_t m = __ldg(p.mask + g);
      const int my_slot = slot_on_lane_rank(p, g, s, t, m, lane);
      if (seg == 0) write_meta_2d(p, g, s, t, m, my_slot, lane);
      for (uint32_t mm = m; mm; mm &= mm - 1) {
        const int r = __ffs(mm) - 1;
        const int sl = __shfl_sync(kFull, my_slot, r);
        uint8_t* dst = p.out_x + ((int64_t)r * p.cap + sl) * p.out_row_bytes;
#pragma unroll
        for (int i = 0; i < kCopyUnroll; ++i) {
          const int64_t off = ((int64_t)seg * kCopyUnroll + i) * 512 + lane * 16;
          if (off < p.in_row_bytes) st_v4(dst + off, v[i]);
        }
      }
    } else {
      const int64_t my_row = row_on_lane_slot(p, g, s, t, lane);
      if (seg == 0) write_meta_std(p, g, s, t, my_row, lane);
      for (uint32_t mm = __ballot_sync(kFull, my_row >= 0); mm; mm &= mm - 1) {
        const int j = __ffs(mm) - 1;
        const int64_t row = __shfl_sync(kFull, my_row, j);
        uint8_t* dst = p.out_x + row * p.out_row_bytes;
#pragma unroll
        for (int i = 0; i < kCopyUnroll; ++i) {
          const int64_t off = ((int64_t)seg * kCopyUnroll + i) * 512 + lane * 16;
          if (off < p.in_row_bytes) st_v4(dst + off, v[i]);
        }
      }
    }
  }
  pdl_wait();  // never finish before the routing layout, even with no work
  if (!STD) recv_from_counts(p);
}

// ------------------------------------------------------------ FP8 quant mode
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
  uint32_t c[8];
  if (amax == 0.f) {
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
  uint32_t out[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = bf16_lo(w[4 * h + j]);
      f[2 * j + 1] = bf16_hi(w[4 * h + j]);
    }
    if (amax != 0.f) {
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = __fdiv_rn(f[j], scale);
    }
    out[h] = cvt_e2m1x8(f);
  }
  q = make_uint4(out[0], out[1], out[2], out[3]);
}

template <bool STD, bool FP4>
__global__ void __launch_bounds__(256, 4) dispatch_quant_kernel(DispatchParams p) {
  const int lane = threadIdx.x & 31;
  const int nb = p.H / (FP4 ? 32 : 128);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  bool waited = false;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < p.total_units;
       u += nwarps) {
    const int64_t g = u / p.segs_per_token;
    const int seg = (int)(u - g * p.segs_per_token);
    const int s = (int)(g / p.Tmax), t = (int)(g - (int64_t)s * p.Tmax);
    if (t >= p.ntok[s]) continue;

    const uint8_t* src = p.x + g * p.in_row_bytes;
    uint4 q[kQuantUnroll];
    float sc[kQuantUnroll];
    // FP4: lane covers elements e32 .. e32 + 31 of the unit's 1024
    const int e32 = seg * (kQuantUnroll * 512) + lane * 32;
    if (FP4) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[i] = e32 < p.H ? ld_nc_v4(src + (int64_t)e32 * 2 + 16 * i) : make_uint4(0, 0, 0, 0);
      quant32_fp4(v, q[0], sc[0]);
    } else {
      uint4 a[kQuantUnroll], b[kQuantUnroll];
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int e0 = (seg * kQuantUnroll + i) * 512 + lane * 16;
        if (e0 < p.H) {
          a[i] = ld_nc_v4(src + (int64_t)e0 * 2);
          b[i] = ld_nc_v4(src + (int64_t)e0 * 2 + 16);
        } else {
          a[i] = make_uint4(0, 0, 0, 0);
          b[i] = a[i];
        }
      }
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) quant16(a[i], b[i], q[i], sc[i]);
      // the unit's 8 block scales sit in lanes 0, 8, 16, 24 (two each): move
      // scale j to lane j so each destination takes them in one store
      static_assert(kQuantUnroll == 2, "scale gather assumes two 512-element steps");
      const int from = (lane & 3) * 8;
      const float s0 = __shfl_sync(kFull, sc[0], from), s1 = __shfl_sync(kFull, sc[1], from);
      sc[0] = lane < 4 ? s0 : s1;
    }
    if (!waited) {  // the routing layout is complete and visible past this point
      pdl_wait();
      waited = true;
    }

    // Each destination row gets the codes and the block scales.
    auto put = [&](int64_t row) {
      uint8_t* dst = p.out_x + row * p.out_row_bytes;
      float* dsc = reinterpret_cast<float*>(p.out_scales) + row * nb;
      if (FP4) {
        if (e32 < p.H) {
          st_v4(dst + e32 / 2, q[0]);
          dsc[e32 / 32] = sc[0];
        }
      } else {
#pragma unroll
        for (int i = 0; i < kQuantUnroll; ++i) {
          const int e0 = (seg * kQuantUnroll + i) * 512 + lane * 16;
          if (e0 < p.H) st_v4(dst + e0, q[i]);
        }
        const int blk = seg * (kQuantUnroll * 4) + lane;  // lanes 0..7: the unit's blocks
        if (lane < kQuantUnroll * 4 && blk * 128 < p.H) dsc[blk] = sc[0];
      }
    };
    if (!STD) {
      const uint32_t m = __ldg(p.mask + g);
      const int my_slot = slot_on_lane_rank(p, g, s, t, m, lane);
      if (seg == 0) write_meta_2d(p, g, s, t, m, my_slot, lane);
      for (uint32_t mm = m; mm; mm &= mm - 1) {
        const int r = __ffs(mm) - 1;
        const int sl = __shfl_sync(kFull, my_slot, r);
        put((int64_t)r * p.cap + sl);
      }
    } else {
      const int64_t my_row = row_on_lane_slot(p, g, s, t, lane);
      if (seg == 0) write_meta_std(p, g, s, t, my_row, lane);
      for (uint32_t mm = __ballot_sync(kFull, my_row >= 0); mm; mm &= mm - 1) {
        const int j = __ffs(mm) - 1;
        put(__shfl_sync(kFull, my_row, j));
      }
    }
  }
  pdl_wait();  // never finish before the routing layout, even with no work
  if (!STD) recv_from_counts(p);
}

template <bool STD>
cudaError_t launch_dispatch(const DispatchParams& p, int quant, const LaunchCfg& lc,
                            cudaStream_t st) {
  if (p.total_units == 0) return cudaSuccess;
  auto k = quant == EP_QUANT_FP8_E4M3_BLOCK128  ? dispatch_quant_kernel<STD, false>
           : quant == EP_QUANT_FP4_E2M1_BLOCK32 ? dispatch_quant_kernel<STD, true>
                                                : dispatch_copy_kernel<STD>;
  return launch_pdl(k, auto_grid(k, lc, p.total_units), lc.block, 0, st, p);
}

}  // namespace

cudaError_t launch_dispatch_2d(const DispatchParams& p, int quant, const LaunchCfg& lc,
                               cudaStream_t st) {
  return launch_dispatch<false>(p, quant, lc, st);
}

cudaError_t launch_dispatch_std(const DispatchParams& p, int quant, const LaunchCfg& lc,
                                cudaStream_t st) {
  return launch_dispatch<true>(p, quant, lc, st);
}

}  // namespace ep

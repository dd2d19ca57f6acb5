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
#include "ep_dispatch_common.cuh"

namespace ep {
namespace {

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

// ---------------------------------------------------- FP8 / FP4 quant mode
// bf16 in; the block quantisers (quant16, quant32_fp4) live in
// ep_dispatch_common.cuh.

// RCP (FP8): quotients from the block scale's reciprocal (fewer instructions;
// faster for small batches, slower for large FP8 ones on GB300); FP4 always
// uses it.
template <bool STD, bool FP4, bool RCP>
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
      for (int i = 0; i < kQuantUnroll; ++i) quant16<RCP>(a[i], b[i], q[i], sc[i]);
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

// FP8 dispatch takes the reciprocal-and-residual quotients below this many
// source tokens (measured on GB300: 8 % faster at 1024 tokens, 3 % at 4096, 4-8 %
// slower from 8192 tokens on), IEEE division from there.
constexpr int64_t kRcpQuotientMaxTokens = 8192;

template <bool STD>
cudaError_t launch_dispatch(const DispatchParams& p, int quant, const LaunchCfg& lc,
                            cudaStream_t st) {
  if (p.total_units == 0) return cudaSuccess;
  int64_t tokens = 0;
  for (int s = 0; s < p.R; ++s) tokens += p.ntok[s];
  auto k = quant == EP_QUANT_FP8_E4M3_BLOCK128
               ? (tokens < kRcpQuotientMaxTokens ? dispatch_quant_kernel<STD, false, true>
                                                 : dispatch_quant_kernel<STD, false, false>)
           : quant == EP_QUANT_FP4_E2M1_BLOCK32 ? dispatch_quant_kernel<STD, true, true>
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

// Device helpers shared by the gather kernels (combine and the split-phase
// combine_recv): 8-element row loads, stores and the fixed-order reduction of
// a token's rows (MORI-EP User Guide, section 3, combine()).
#pragma once

#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr int kVec = 8;  // elements per lane per 256-element step

// Load 8 consecutive elements as f32.
template <int DT>
__device__ __forceinline__ void load8(const uint8_t* base, int64_t elem, float f[8]) {
  if (DT == EP_DTYPE_BF16) {
    const uint4 v = ld_nc_v4(base + elem * 2);
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  } else {
    const uint4 a = ld_nc_v4(base + elem * 4);
    const uint4 b = ld_nc_v4(base + elem * 4 + 16);
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
    f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
  }
}

// Raw 16-byte loads of 8 elements (one vector for bf16, two for f32).
template <int DT>
struct Raw8 {
  uint4 a, b;
};

template <int DT>
__device__ __forceinline__ Raw8<DT> load_raw8(const uint8_t* base, int64_t elem) {
  Raw8<DT> r;
  if (DT == EP_DTYPE_BF16) {
    r.a = ld_nc_v4(base + elem * 2);
  } else {
    r.a = ld_nc_v4(base + elem * 4);
    r.b = ld_nc_v4(base + elem * 4 + 16);
  }
  return r;
}

template <int DT>
__device__ __forceinline__ void unpack8(const Raw8<DT>& r, float f[8]) {
  if (DT == EP_DTYPE_BF16) {
    f[0] = bf16_lo(r.a.x); f[1] = bf16_hi(r.a.x); f[2] = bf16_lo(r.a.y); f[3] = bf16_hi(r.a.y);
    f[4] = bf16_lo(r.a.z); f[5] = bf16_hi(r.a.z); f[6] = bf16_lo(r.a.w); f[7] = bf16_hi(r.a.w);
  } else {
    f[0] = __uint_as_float(r.a.x); f[1] = __uint_as_float(r.a.y);
    f[2] = __uint_as_float(r.a.z); f[3] = __uint_as_float(r.a.w);
    f[4] = __uint_as_float(r.b.x); f[5] = __uint_as_float(r.b.y);
    f[6] = __uint_as_float(r.b.z); f[7] = __uint_as_float(r.b.w);
  }
}

template <int DT>
__device__ __forceinline__ void store8(uint8_t* base, int64_t elem, const float f[8]) {
  if (DT == EP_DTYPE_BF16) {
    uint4 v;
    v.x = cvt_bf16x2(f[0], f[1]);
    v.y = cvt_bf16x2(f[2], f[3]);
    v.z = cvt_bf16x2(f[4], f[5]);
    v.w = cvt_bf16x2(f[6], f[7]);
    st_v4_cs(base + elem * 2, v);
  } else {
    st_v4_cs(base + elem * 4, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                      __float_as_uint(f[2]), __float_as_uint(f[3])));
    st_v4_cs(base + elem * 4 + 16, make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]),
                                           __float_as_uint(f[6]), __float_as_uint(f[7])));
  }
}

constexpr int dt_size(int dt) { return dt == EP_DTYPE_BF16 ? 2 : 4; }

// Reduce the D rows at ptr[0..D) (already in reduction order) for this unit.
// MAXD > 0: rows held in registers, all loads of the unit issued up front.
template <int IN, int OUT, int MAXD>
__device__ __forceinline__ void reduce_rows(const CombineParams& p, const uint8_t* const* ptr,
                                            const float* wd, int D, int seg, int lane,
                                            uint8_t* out_row) {
  if (MAXD > 0) {
    Raw8<IN> v[kCombineUnroll][MAXD > 0 ? MAXD : 1];
#pragma unroll
    for (int i = 0; i < kCombineUnroll; ++i) {
      const int e0 = (seg * kCombineUnroll + i) * 256 + lane * kVec;
#pragma unroll
      for (int d = 0; d < MAXD; ++d)
        if (d < D && e0 < p.H) v[i][d] = load_raw8<IN>(ptr[d], e0);
    }
#pragma unroll
    for (int i = 0; i < kCombineUnroll; ++i) {
      const int e0 = (seg * kCombineUnroll + i) * 256 + lane * kVec;
      if (e0 >= p.H) continue;
      float acc[kVec];
#pragma unroll
      for (int q = 0; q < kVec; ++q) acc[q] = 0.0f;
#pragma unroll
      for (int d = 0; d < MAXD; ++d) {
        if (d < D) {
          float f[kVec];
          unpack8<IN>(v[i][d], f);
#pragma unroll
          for (int q = 0; q < kVec; ++q)
            acc[q] = p.weighted ? __fmaf_rn(wd[d], f[q], acc[q]) : __fadd_rn(acc[q], f[q]);
        }
      }
      store8<OUT>(out_row, e0, acc);
    }
  } else {
#pragma unroll
    for (int i = 0; i < kCombineUnroll; ++i) {
      const int e0 = (seg * kCombineUnroll + i) * 256 + lane * kVec;
      if (e0 >= p.H) continue;
      float acc[kVec];
#pragma unroll
      for (int q = 0; q < kVec; ++q) acc[q] = 0.0f;
      for (int d = 0; d < D; ++d) {
        float f[kVec];
        load8<IN>(ptr[d], e0, f);
#pragma unroll
        for (int q = 0; q < kVec; ++q)
          acc[q] = p.weighted ? __fmaf_rn(wd[d], f[q], acc[q]) : __fadd_rn(acc[q], f[q]);
      }
      store8<OUT>(out_row, e0, acc);
    }
  }
}

}  // namespace
}  // namespace ep

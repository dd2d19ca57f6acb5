// Combine: gather expert outputs back to their source tokens and reduce.
//
// MORI-EP User Guide, section 3, combine(): expert outputs return to the
// token's original position; "Choosing an EP API and backend" names the
// HIP backend's combine a gather in BF16/FP32. Here each (token, column
// segment) unit is owned by one warp that reads the token's rows from every
// destination rank holding a copy and reduces them in an f32 accumulator in
// ascending rank order, then rounds once. The fixed order makes the result
// bit-reproducible and independent of scheduling. Weighted mode multiplies
// each rank's row by the sum of the token's weights on that rank (fused
// multiply-add per rank). combine_weights is the weight row of the copy on
// the lowest destination rank.
//
// combine_standard_moe() (section 4) reads one packed row per valid (token,
// slot) instead, in (owner rank, slot) order, weighted by the token's own
// router weights.
#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
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

template <int IN, int OUT, int MAXD>
__global__ void __launch_bounds__(256) combine_2d_kernel(CombineParams p) {
  constexpr int kSlots = MAXD > 0 ? MAXD : EP_MAX_WORLD_SIZE;
  const int lane = threadIdx.x & 31;
  const int64_t in_row = (int64_t)p.H * dt_size(IN);
  const int64_t out_row = (int64_t)p.H * dt_size(OUT);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < p.total_units;
       u += nwarps) {
    const int64_t g = u / p.segs_per_token;
    const int seg = (int)(u - g * p.segs_per_token);
    const int s = (int)(g / p.Tmax), t = (int)(g - (int64_t)s * p.Tmax);
    if (t >= p.ntok[s]) continue;

    const int sl = lane < p.R ? __ldg(p.slot_map + g * p.R + lane) : -1;
    const uint32_t m = __ballot_sync(kFull, sl >= 0);
    const int D = __popc(m);
    float wr = 0.0f;
    if (p.weighted && sl >= 0) {
      const int64_t row = (int64_t)lane * p.cap + sl;
      for (int j = 0; j < p.k; ++j) {
        const int e = __ldg(p.recv_idx + row * p.k + j);
        if (e >= 0 && e / p.E_r == lane) wr = __fadd_rn(wr, __ldg(p.w + row * p.k + j));
      }
    }
    if (seg == 0 && p.out_w) {
      const int rmin = m ? __ffs(m) - 1 : 0;
      const int slmin = __shfl_sync(kFull, sl, rmin);
      if (lane < p.k)
        p.out_w[g * p.k + lane] =
            m ? __ldg(p.w + ((int64_t)rmin * p.cap + slmin) * p.k + lane) : 0.0f;
    }
    const uint8_t* ptr[kSlots];
    float wd[kSlots];
    uint32_t mm = m;
#pragma unroll
    for (int d = 0; d < kSlots; ++d) {
      const int r = mm ? __ffs(mm) - 1 : 0;
      mm &= mm - 1;
      const int sld = __shfl_sync(kFull, sl, r);
      ptr[d] = p.y + ((int64_t)r * p.cap + (sld < 0 ? 0 : sld)) * in_row;
      wd[d] = __shfl_sync(kFull, wr, r);
    }
    reduce_rows<IN, OUT, MAXD>(p, ptr, wd, D, seg, lane, p.out + g * out_row);
  }
}

template <int IN, int OUT, int MAXD>
__global__ void __launch_bounds__(256) combine_std_kernel(CombineParams p) {
  constexpr int kSlots = MAXD > 0 ? MAXD : EP_MAX_TOPK;
  const int lane = threadIdx.x & 31;
  const int64_t in_row = (int64_t)p.H * dt_size(IN);
  const int64_t out_row = (int64_t)p.H * dt_size(OUT);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // packed row of slot `lane` of unit u's token (-1: none)
  auto row_of = [&](int64_t u) -> int {
    if (u >= p.total_units || lane >= p.k) return -1;
    const int64_t g = u / p.segs_per_token;
    const int s = (int)(g / p.Tmax), t = (int)(g - (int64_t)s * p.Tmax);
    return t < p.ntok[s] ? __ldg(p.row_map + g * p.k + lane) : -1;
  };
  int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int row_next = row_of(u);
  for (; u < p.total_units; u += nwarps) {
    const int row = row_next;
    row_next = row_of(u + nwarps);  // prefetch: overlaps this unit's row loads
    const int64_t g = u / p.segs_per_token;
    const int seg = (int)(u - g * p.segs_per_token);
    const int s = (int)(g / p.Tmax), t = (int)(g - (int64_t)s * p.Tmax);
    if (t >= p.ntok[s]) continue;

    const bool valid = row >= 0;
    const int key = valid ? (int)(row / p.cap) * 32 + lane : 0x7FFFFFFF;
    const float wj = (valid && p.weighted) ? __ldg(p.w + g * p.k + lane) : 0.0f;
    // position of this slot in (owner rank, slot) order
    int pos = 0;
    for (int i = 0; i < p.k; ++i) pos += __shfl_sync(kFull, key, i) < key;
    const uint32_t vm = __ballot_sync(kFull, valid);
    const int D = __popc(vm);
    const uint8_t* ptr[kSlots];
    float wd[kSlots];
#pragma unroll
    for (int d = 0; d < kSlots; ++d) {
      const uint32_t b = __ballot_sync(kFull, valid && pos == d);
      const int j = b ? __ffs(b) - 1 : 0;
      const int rd = __shfl_sync(kFull, row, j);
      ptr[d] = p.y + (int64_t)(rd < 0 ? 0 : rd) * in_row;
      wd[d] = __shfl_sync(kFull, wj, j);
    }
    reduce_rows<IN, OUT, MAXD>(p, ptr, wd, D, seg, lane, p.out + g * out_row);
  }
}

template <template <int, int, int> class KSel, int MAXD_SMALL>
cudaError_t launch_combine(const CombineParams& p, int in_dtype, int out_dtype, bool small,
                           const LaunchCfg& lc, cudaStream_t st) {
  if (p.total_units == 0) return cudaSuccess;
  cudaError_t err = cudaSuccess;
  auto go = [&](auto kernel) {
    kernel<<<auto_grid(kernel, lc, p.total_units), lc.block, 0, st>>>(p);
    err = cudaGetLastError();
  };
  const bool ib = in_dtype == EP_DTYPE_BF16, ob = out_dtype == EP_DTYPE_BF16;
  if (ib && ob) small ? go(KSel<EP_DTYPE_BF16, EP_DTYPE_BF16, MAXD_SMALL>::fn) : go(KSel<EP_DTYPE_BF16, EP_DTYPE_BF16, 0>::fn);
  else if (ib) small ? go(KSel<EP_DTYPE_BF16, EP_DTYPE_FP32, MAXD_SMALL>::fn) : go(KSel<EP_DTYPE_BF16, EP_DTYPE_FP32, 0>::fn);
  else if (ob) small ? go(KSel<EP_DTYPE_FP32, EP_DTYPE_BF16, MAXD_SMALL>::fn) : go(KSel<EP_DTYPE_FP32, EP_DTYPE_BF16, 0>::fn);
  else small ? go(KSel<EP_DTYPE_FP32, EP_DTYPE_FP32, MAXD_SMALL>::fn) : go(KSel<EP_DTYPE_FP32, EP_DTYPE_FP32, 0>::fn);
  return err;
}

template <int IN, int OUT, int MAXD>
struct Sel2d {
  static constexpr auto fn = combine_2d_kernel<IN, OUT, MAXD>;
};
template <int IN, int OUT, int MAXD>
struct SelStd {
  static constexpr auto fn = combine_std_kernel<IN, OUT, MAXD>;
};

}  // namespace

cudaError_t launch_combine_2d(const CombineParams& p, int in_dtype, int out_dtype,
                              const LaunchCfg& lc, cudaStream_t st) {
  return launch_combine<Sel2d, 8>(p, in_dtype, out_dtype, p.R <= 8, lc, st);
}

cudaError_t launch_combine_std(const CombineParams& p, int in_dtype, int out_dtype,
                               const LaunchCfg& lc, cudaStream_t st) {
  return launch_combine<SelStd, 8>(p, in_dtype, out_dtype, p.k <= 8, lc, st);
}

}  // namespace ep

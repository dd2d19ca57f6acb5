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
#include "ep_combine_common.cuh"

namespace ep {
namespace {

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
  // first pool row of each rank: the owner rank of a pool row is the last
  // rank whose region starts at or before it
  __shared__ int base[EP_MAX_WORLD_SIZE];
  if ((int)threadIdx.x < p.R) base[threadIdx.x] = __ldg(p.rank_base + threadIdx.x);
  __syncthreads();
  auto owner = [&](int row) {
    int r = 0;
    while (r + 1 < p.R && row >= base[r + 1]) ++r;
    return r;
  };
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
    const int key = valid ? owner(row) * 32 + lane : 0x7FFFFFFF;
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

// Copy-mode dispatch with bulk asynchronous copies (the TMA engine).
//
// Same results as dispatch_copy_kernel (MORI-EP User Guide, section 3,
// dispatch(); section 4, dispatch_standard_moe()): payload bits move
// unchanged. One warp per CTA takes whole tokens. Lane 0 keeps a ring of
// four shared-memory stages filled with source rows (one cp.async.bulk
// global->shared per row, completing on the stage's mbarrier) and writes
// each arrived row to every destination with one cp.async.bulk
// shared->global per destination; a stage is refilled once the stores that
// read it have finished reading. The other lanes compute the destinations
// and write the per-row metadata with ordinary stores. Row loads are issued
// before waiting for the routing layout (programmatic dependent launch), so
// they overlap it. Waits on mbarriers are bounded (error bit on timeout).
#include "ep_bulk.cuh"
#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr int kStages = 4;

struct BulkRing {
  uint64_t full[kStages];
};

template <bool STD>
__global__ void __launch_bounds__(32) dispatch_bulk_copy_kernel(DispatchParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  BulkRing& ring = *reinterpret_cast<BulkRing*>(smem_raw);
  uint8_t* rows = smem_raw + 128;                 // kStages x in_row_bytes
  const int lane = threadIdx.x;
  const uint32_t rb = (uint32_t)p.in_row_bytes;
  const int64_t ntokens = (int64_t)p.R * p.Tmax;
  auto present = [&](int64_t g) {
    const int s = (int)(g / p.Tmax);
    return (int)(g - (int64_t)s * p.Tmax) < p.ntok[s];
  };
  // the n-th present token of this CTA, starting the search at g
  auto next_present = [&](int64_t g) {
    while (g < ntokens && !present(g)) g += gridDim.x;
    return g;
  };
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&ring.full[s], 1);
    mbar_init_fence();
  }
  __syncwarp();

  // prologue: the first kStages rows of this CTA. Load j (the CTA's j-th
  // present token) lands in stage j % kStages, phase (j / kStages) & 1.
  int issued = 0;
  int64_t load_g = next_present(blockIdx.x);
  for (int s = 0; s < kStages && load_g < ntokens; ++s) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&ring.full[s], rb);
      bulk_g2s(rows + (size_t)s * rb, p.x + load_g * p.in_row_bytes, rb, &ring.full[s]);
    }
    ++issued;
    load_g = next_present(load_g + gridDim.x);
  }
  pdl_wait();  // the routing layout is complete and visible past this point

  int i = 0;
  bool ok = true;
  for (int64_t g = next_present(blockIdx.x); g < ntokens; g = next_present(g + gridDim.x), ++i) {
    const int st = i % kStages;
    const int s = (int)(g / p.Tmax), t = (int)(g - (int64_t)s * p.Tmax);
    // destinations: receive slot on rank `lane` (2D) or packed row of slot `lane`
    int64_t dst_row = -1;
    uint32_t m;
    if (!STD) {
      const uint32_t mask = __ldg(p.mask + g);
      int sl = -1;
      if (lane < p.R && ((mask >> lane) & 1u)) {
        const int c = s * p.cpr + t / kChunk;
        sl = __ldg(p.chunk_off + (int64_t)c * p.R + lane) + (int)__ldg(p.local8 + g * p.R + lane);
        dst_row = (int64_t)lane * p.cap + sl;
        p.src_pos[dst_row] = s * (p.R * p.Tmax) + t;
      }
      if (lane < p.R) p.slot_map[g * p.R + lane] = sl;
      m = __ballot_sync(kFull, dst_row >= 0);
      const float wv = lane < p.k ? __ldg(p.w + g * p.k + lane) : 0.f;
      const int iv = lane < p.k ? __ldg(p.idx + g * p.k + lane) : 0;
      for (uint32_t mm = m; mm; mm &= mm - 1) {
        const int64_t row = __shfl_sync(kFull, dst_row, __ffs(mm) - 1);
        if (lane < p.k) {
          p.out_w[row * p.k + lane] = wv;
          p.out_idx[row * p.k + lane] = iv;
        }
      }
    } else {
      if (lane < p.k) {
        const int e = __ldg(p.idx + g * p.k + lane);
        const int l = __ldg(p.local16 + g * p.k + lane);
        if (e >= 0 && e < p.E && l != 0xFFFF) {
          const int c = s * p.cpr + t / kChunk;
          const int64_t row = (int64_t)__ldg(p.rank_base + e / p.E_r) +
                              __ldg(p.expert_offset + e) +
                              __ldg(p.chunk_off + (int64_t)c * p.E + e) + l;
          if (row < p.cap) dst_row = row;
        }
        p.row_map[g * p.k + lane] = (int32_t)dst_row;
        if (dst_row >= 0) p.src_pos[dst_row] = s * (p.R * p.Tmax) + t;
      }
      m = __ballot_sync(kFull, dst_row >= 0);
    }
    if (p.scale_row_bytes > 0 && p.scales_in) {
      for (uint32_t mm = m; mm; mm &= mm - 1) {
        const int64_t row = __shfl_sync(kFull, dst_row, __ffs(mm) - 1);
        const uint8_t* src = p.scales_in + g * p.scale_row_bytes;
        uint8_t* dst = p.out_scales + row * p.scale_row_bytes;
        for (int q = lane; q < p.scale_row_bytes; q += 32) dst[q] = __ldg(src + q);
      }
    }
    // payload: wait for the row, then one bulk store per destination
    if (lane == 0) ok = mbar_wait(&ring.full[st], (uint32_t)(i / kStages) & 1u);
    ok = __shfl_sync(kFull, ok, 0);
    if (!ok) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      break;
    }
    for (uint32_t mm = m; mm; mm &= mm - 1) {
      const int64_t row = __shfl_sync(kFull, dst_row, __ffs(mm) - 1);
      if (lane == 0) bulk_s2g(p.out_x + row * p.out_row_bytes, rows + (size_t)st * rb, rb);
    }
    if (lane == 0) {
      bulk_commit();
      // refill the previous token's stage once its stores have read it
      if (i >= 1 && load_g < ntokens) {
        bulk_wait_read<1>();
        const int ps = (i - 1) % kStages;
        mbar_arrive_expect_tx(&ring.full[ps], rb);
        bulk_g2s(rows + (size_t)ps * rb, p.x + load_g * p.in_row_bytes, rb, &ring.full[ps]);
      }
    }
    if (i >= 1 && load_g < ntokens) ++issued;
    if (i >= 1) load_g = __shfl_sync(kFull, load_g < ntokens ? next_present(load_g + gridDim.x)
                                                             : load_g, 0);
  }
  if (lane == 0) {
    // no copy may still read or write this CTA's shared memory when it exits:
    // the stores are drained by the bulk group wait; after a timeout, the
    // row loads issued for tokens i .. issued-1 are waited for as well (all
    // of those waits together bounded by about a second)
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (!ok) {
      const uint64_t t0 = globaltimer_ns();
      for (int j = i; j < issued; ++j)
        while (!mbar_try_wait(&ring.full[j % kStages], (uint32_t)(j / kStages) & 1u))
          if (globaltimer_ns() - t0 > kMbarWaitNs) break;
    }
  }
}

// Failure-detection self-test: one thread waits on an mbarrier that nothing
// ever completes. The bounded wait gives up after about a second and the
// kernel records the timeout bit, as every bulk kernel does, then returns
// normally (no trap, no fault; the context stays usable).
__global__ void bounded_wait_selftest_kernel(int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
    if (!mbar_wait(&bar, 0)) atomicOr(err, kErrTimeout);
  }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int32_t* err, cudaStream_t st) {
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(err);
  return cudaGetLastError();
}

bool dispatch_bulk_supported(const DispatchParams& p) {
  return p.in_row_bytes <= 48 * 1024 && p.in_row_bytes % 16 == 0;
}

cudaError_t launch_dispatch_bulk_copy(const DispatchParams& p, bool std_layout,
                                      const LaunchCfg& lc, cudaStream_t st) {
  const int64_t ntokens = (int64_t)p.R * p.Tmax;
  if (ntokens == 0) return cudaSuccess;
  auto k = std_layout ? dispatch_bulk_copy_kernel<true> : dispatch_bulk_copy_kernel<false>;
  const size_t smem = 128 + (size_t)kStages * p.in_row_bytes;
  const int per_sm = ctas_per_sm(k, 32, smem);  // also raises the smem limit
  // default: one resident wave; for the packed layout, whose tokens carry
  // very different row counts, several waves (8 CTAs per SM requested) so
  // CTAs that finish early hand their SM to the next ones (measured on GB300:
  // 9 % faster for Zipf-skewed routing, 2 % slower for the 2D layout)
  int64_t grid = lc.grid_hint > 0 ? lc.grid_hint
                                  : (int64_t)lc.sm_count * (std_layout && per_sm < 8 ? 8 : per_sm);
  if (grid > ntokens) grid = ntokens;
  return launch_pdl(k, (int)grid, 32, smem, st, p);
}

}  // namespace ep

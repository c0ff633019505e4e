// Persistent grouped GEMM of MXFP8 grouped-matmul-finalize-routing on sm_103a.
//
// Work: for every token group g (at most TMAX routed tokens of one expert e),
// every 128-column tile j of the output and every 128-element K block kb,
//   D[n, t] += sum_{k in block} (x2[e,k,n] * s_w) * (x1[t,k] * s_x)
// with tcgen05.mma kind::mxf8f6f4 block_scale (one E8M0 scale per 32 K).
// The weights are the 128-row A operand (rows = output columns), the tokens the
// N-wide B operand (N = tokens rounded up to 16), so experts holding few tokens
// still stream each weight byte exactly once.
//
// Roles (192 threads, one CTA per SM):
//   warp 0     TMA producer: prepared weight tile + its scales (one bulk copy),
//              token rows (16-row tensor-map boxes), token scales (bulk copy)
//   warp 1     TMEM owner and MMA issuer (scale copies to TMEM, 4 MMAs per stage)
//   warps 2-5  epilogue: TMEM -> registers, x logit, red.global.add.f32 into
//              out[row_index[t], n] (or a plain store into the per-token buffer in
//              deterministic mode); before the first tile they add the shared
//              input for their slice of rows.
//
// Scheduling: atomic mode splits the total (group, tile, K-block) iteration space
// evenly over the CTAs (stream-K); a tile cut between CTAs is finished by
// atomics, which is exact up to FP32 rounding order since every term is linear.
// Deterministic mode gives each (group, tile, K-split) unit to one CTA and
// stores its result for the row-ordered combine.
//
// Every wait is bounded: on timeout the CTA sets GMMFR_DEV_TIMEOUT, stops
// issuing, waits (bounded) for its copies and MMAs in flight, frees TMEM and exits.
#include "common.cuh"
#include "ptx.cuh"

namespace gmmfr {

template <int TMAX>
struct GemmCfg {
  static constexpr int kXBytes = TMAX * 128;
  static constexpr int kOffW = 0;                        // 16384 B weights (1024-aligned)
  static constexpr int kOffWSF = kWTileBytes;            // 512 B weight scales
  static constexpr int kOffXSF = kWTileBytes + kSfChunk; // 512 B token scales
  static constexpr int kOffX = kWTileBytes + 2 * kSfChunk;  // token rows (1024-aligned)
  static constexpr int kStageBytes = kOffX + kXBytes;
  static constexpr int kStages = TMAX == 128 ? 6 : (TMAX == 64 ? 8 : 10);
  static constexpr int kSfCol0 = 2 * TMAX;  // TMEM: 2 accumulators, then 8 scale columns per stage
  static constexpr int kTmemCols = (2 * TMAX + 8 * kStages) <= 256 ? 256 : 512;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = kStages * kStageBytes + kBarBytes + 1024;
  static_assert(kOffX % 1024 == 0 && kStageBytes % 1024 == 0, "operand tiles must stay 1024-aligned");
  static_assert(2 * TMAX + 8 * kStages <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Seg {
  int g, j, kb0, kb1, slot;
};

// The sequence of (group, tile, K range) segments of one CTA; every role walks it.
// Tiles are ordered column-tile-major (tile = j * n_groups + g), so the token
// groups of one expert that holds more than TMAX tokens are adjacent and their
// shared weight tiles are re-read while still in L2.
struct Sched {
  int64_t i, i_end, step;
  int NT, KB, split, ng;
  bool det;
  __device__ void init(int n_groups, int NT_, int KB_, bool det_, int split_) {
    ng = n_groups;
    NT = NT_;
    KB = KB_;
    det = det_;
    split = split_;
    const int64_t tiles = (int64_t)n_groups * NT;
    if (!det) {
      const int64_t total = tiles * KB;
      i = total * blockIdx.x / gridDim.x;
      i_end = total * (blockIdx.x + 1) / gridDim.x;
      step = 0;
    } else {
      i = blockIdx.x;
      i_end = tiles * split;
      step = gridDim.x;
    }
  }
  __device__ bool next(Seg& s) {
    if (i >= i_end) return false;
    int64_t tile;
    if (!det) {
      tile = i / KB;
      s.kb0 = (int)(i % KB);
      const int64_t left = i_end - i;
      s.kb1 = (int)((KB - s.kb0) < left ? KB : s.kb0 + left);
      i += s.kb1 - s.kb0;
      s.slot = 0;
    } else {
      tile = i / split;
      const int sp = (int)(i % split);
      s.kb0 = (int)((int64_t)sp * KB / split);
      s.kb1 = (int)((int64_t)(sp + 1) * KB / split);
      s.slot = sp;
      i += step;
    }
    s.g = (int)(tile % ng);
    s.j = (int)(tile / ng);
    return true;
  }
};

struct Ctl {
  volatile int* abort;
  uint32_t* err;
  int64_t timeout_ns;
};

// Bounded wait for the phase of `parity` to complete.  Gives up when another
// role aborted or after timeout_ns (then records the timeout and aborts).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (ptx::globaltimer() - t0 > (uint64_t)c.timeout_ns) {
      *c.abort = 1;
      atomicOr(c.err, kErrTimeout);
      return false;
    }
  }
}

// Wait used while draining after an abort: ignores the abort flag, fixed 1 s limit.
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > 1000000000ull) return false;
  }
  return true;
}

__device__ __forceinline__ int load_row32(const void* rows, int row_i32, int64_t t, int64_t batch) {
  const int64_t r = row_i32 ? (int64_t) static_cast<const int32_t*>(rows)[t] : static_cast<const int64_t*>(rows)[t];
  return (r >= 0 && r < batch) ? (int)r : -1;
}

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// out[offset + i, n] += w * shared[i, n] for this CTA's slice (atomic mode only).
__device__ void shared_add_slice(const GemmParams& p, int ep_tid) {
  const int64_t R = p.shared_rows, N = p.N;
  const bool vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.out) & 15) == 0) &&
                   ((reinterpret_cast<uintptr_t>(p.shared) & 7) == 0);
  if (vec) {
    const int64_t n4 = N / 4, total = R * n4;
    const int64_t a = total * blockIdx.x / gridDim.x, b = total * (blockIdx.x + 1) / gridDim.x;
    for (int64_t idx = a + ep_tid; idx < b; idx += 128) {
      const int64_t i = idx / n4, n = (idx % n4) * 4;
      const uint2 raw = *reinterpret_cast<const uint2*>(p.shared + i * N + n);
      const float w = p.shared_weight;
      ptx::red_add_v4_f32(p.out + (p.shared_offset + i) * N + n, w * bf16f(raw.x & 0xFFFF), w * bf16f(raw.x >> 16),
                          w * bf16f(raw.y & 0xFFFF), w * bf16f(raw.y >> 16));
    }
  } else {
    const int64_t total = R * N;
    const int64_t a = total * blockIdx.x / gridDim.x, b = total * (blockIdx.x + 1) / gridDim.x;
    for (int64_t idx = a + ep_tid; idx < b; idx += 128) {
      const int64_t i = idx / N, n = idx % N;
      ptx::red_add_f32(p.out + (p.shared_offset + i) * N + n, p.shared_weight * bf16f(p.shared[i * N + n]));
    }
  }
}

template <int TMAX>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_x1, const __grid_constant__ GemmParams p) {
  using C = GemmCfg<TMAX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* full = bars;                      // [kStages] TMA bytes landed
  uint64_t* empty = bars + C::kStages;        // [kStages] MMAs done reading the stage
  uint64_t* accf = bars + 2 * C::kStages;     // [2] accumulator ready
  uint64_t* acce = accf + 2;                  // [2] accumulator drained by the epilogue
  uint64_t* drain = acce + 2;                 // [1] all MMAs of this CTA complete
  uint64_t* stall = drain + 1;                // [1] never arrived on (testing aid)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stall + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&accf[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&acce[b]), 4);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    ptx::mbar_init(ptx::smem_u32(stall), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) ptx::prefetch_tensormap(&tmap_x1);
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  const int n_groups = (int)p.hdr[kHdrGroups];
  Sched sched;
  sched.init(n_groups, p.NT, p.KB, p.deterministic != 0, p.split);
  const uint32_t smem_base = ptx::smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_stream = ptx::l2_evict_first_policy();  // weights: read once
      const uint64_t pol_keep = ptx::l2_evict_last_policy();     // tokens: reused by every tile
      int fills[C::kStages];
#pragma unroll
      for (int s = 0; s < C::kStages; ++s) fills[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      if (p.test_stall) ok = wait_bar(ptx::smem_u32(stall), 0, ctl);
      Seg sg;
      while (ok && sched.next(sg)) {
        const int4 gr = p.groups[sg.g];
        const int e = gr.x, t0 = gr.y, T = gr.z;
        const int nbox = (T + kTokBox - 1) / kTokBox;
        const uint32_t tx = kPrepTileBytes + kSfChunk + nbox * kTokBox * 128;
        const uint8_t* wsrc = p.prepared + ((int64_t)e * p.NT + sg.j) * p.KB * (int64_t)kPrepTileBytes;
        const uint8_t* ssrc = p.tsf + (int64_t)sg.g * p.KB * kSfChunk;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!wait_bar(ptx::smem_u32(&empty[stage]), phase ^ 1, ctl)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full[stage]);
          const uint32_t sb = smem_base + stage * C::kStageBytes;
          ptx::mbar_arrive_expect_tx(fb, tx);
          ptx::bulk_g2s(sb + C::kOffW, wsrc + (int64_t)kb * kPrepTileBytes, kPrepTileBytes, fb, pol_stream);
          ptx::bulk_g2s(sb + C::kOffXSF, ssrc + (int64_t)kb * kSfChunk, kSfChunk, fb, pol_keep);
          for (int b = 0; b < nbox; ++b)
            ptx::tma_load_2d(sb + C::kOffX + b * kTokBox * 128, &tmap_x1, kb * kTileK, t0 + b * kTokBox, fb, pol_keep);
          ++fills[stage];
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (ok) {
        // all fills consumed: wait until the MMA warp has released every stage
        for (int s = 0; s < C::kStages; ++s)
          if (fills[s] > 0 && !wait_bar(ptx::smem_u32(&empty[s]), (fills[s] - 1) & 1, ctl)) break;
      }
      if (*abort_flag) {
        // aborted: let every issued copy land before shared memory is released
        for (int s = 0; s < C::kStages; ++s)
          if (fills[s] > 0) wait_bar_drain(ptx::smem_u32(&full[s]), (fills[s] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      Seg sg;
      bool ok = true;
      while (ok && sched.next(sg)) {
        const int T = p.groups[sg.g].z;
        const uint32_t npad = (uint32_t)((T + 15) / 16) * 16;
        const uint32_t idesc = p.idesc | ((npad >> 3) << 17);
        const int buf = acc_i & 1;
        const uint32_t aph = (acc_i >> 1) & 1;
        if (!wait_bar(ptx::smem_u32(&acce[buf]), aph ^ 1, ctl)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * TMAX;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!wait_bar(ptx::smem_u32(&full[stage]), phase, ctl)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sb = smem_base + stage * C::kStageBytes;
          const uint32_t sfa = tmem_base + C::kSfCol0 + stage * 8;
          const uint32_t sfb = sfa + 4;
          ptx::tc_cp_sf(sfa, ptx::smem_desc(sb + C::kOffWSF, 0, 128, ptx::kSwizzleNone));
          ptx::tc_cp_sf(sfb, ptx::smem_desc(sb + C::kOffXSF, 0, 128, ptx::kSwizzleNone));
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint64_t adesc = ptx::smem_desc(sb + C::kOffW + 32 * q, 16, 1024, ptx::kSwizzle128B);
            const uint64_t bdesc = ptx::smem_desc(sb + C::kOffX + 32 * q, 16, 1024, ptx::kSwizzle128B);
            const uint32_t id = idesc | ((uint32_t)q << 4) | ((uint32_t)q << 29);
            ptx::tc_mma_mxf8(d_tmem, adesc, bdesc, id, sfa, sfb, (kb > sg.kb0 || q > 0) ? 1u : 0u);
          }
          ptx::tc_commit(ptx::smem_u32(&empty[stage]));
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        ptx::tc_commit(ptx::smem_u32(&accf[buf]));
        ++acc_i;
      }
      // every MMA of this CTA has completed once `drain` fires
      ptx::tc_commit(ptx::smem_u32(drain));
      wait_bar_drain(ptx::smem_u32(drain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int ep_tid = threadIdx.x - 64;
    if (!p.deterministic && p.shared != nullptr && p.shared_rows > 0 && p.N > 0) shared_add_slice(p, ep_tid);
    int acc_i = 0;
    Seg sg;
    while (sched.next(sg)) {
      const int4 gr = p.groups[sg.g];
      const int t0 = gr.y, T = gr.z;
      const int buf = acc_i & 1;
      const uint32_t aph = (acc_i >> 1) & 1;
      if (!wait_bar(ptx::smem_u32(&accf[buf]), aph, ctl)) break;
      ptx::tc_fence_after();
      const int64_t n = (int64_t)sg.j * kTileN + q * 32 + lane;
      const bool n_ok = n < p.N;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * TMAX;
      bool bad_row = false;
      for (int c0 = 0; c0 < T; c0 += 32) {
        const int tok = c0 + lane;
        int my_row = -1;
        float my_lg = 0.f;
        if (tok < T) {
          my_row = load_row32(p.row_index, p.row_i32, (int64_t)t0 + tok, p.batch);
          my_lg = p.logit ? p.logit[t0 + tok] : 1.f;
          bad_row |= my_row < 0;
        }
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + c0, v);
        ptx::tmem_wait_ld();
        if (c0 + 32 >= T) {  // accumulator fully read: hand it back to the MMA warp
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&acce[buf]));
        }
        const int cnt = T - c0 < 32 ? T - c0 : 32;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          if (jj < cnt) {
            const int row = __shfl_sync(0xffffffffu, my_row, jj);
            const float lg = __shfl_sync(0xffffffffu, my_lg, jj);
            const float val = __uint_as_float(v[jj]) * lg;
            if (n_ok) {
              if (p.deterministic) {
                p.ybuf[((int64_t)sg.slot * p.M + t0 + c0 + jj) * p.N + n] = val;
              } else if (row >= 0) {
                ptx::red_add_f32(p.out + (int64_t)row * p.N + n, val);
              }
            }
          }
        }
      }
      if (bad_row) atomicOr(p.err, kErrBadRowIndex);
      ++acc_i;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

int gemm_smem_bytes(int tmax) {
  switch (tmax) {
    case 32: return GemmCfg<32>::kSmemBytes;
    case 64: return GemmCfg<64>::kSmemBytes;
    default: return GemmCfg<128>::kSmemBytes;
  }
}

template <int TMAX>
static cudaError_t launch_t(const CUtensorMap& tmap, const GemmParams& p, int grid, cudaStream_t s) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<TMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GemmCfg<TMAX>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  gemm_kernel<TMAX><<<grid, kGemmThreads, GemmCfg<TMAX>::kSmemBytes, s>>>(tmap, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const CUtensorMap& tmap, const GemmParams& p, int tmax, int grid, cudaStream_t s) {
  switch (tmax) {
    case 32: return launch_t<32>(tmap, p, grid, s);
    case 64: return launch_t<64>(tmap, p, grid, s);
    case 128: return launch_t<128>(tmap, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gmmfr

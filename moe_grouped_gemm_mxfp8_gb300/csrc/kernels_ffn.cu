// Grouped SwiGLU expert FFN in BF16 (llada2_moe_grouped_gemm, LLaDA2.0-mini
// grouped-GEMM write-up, sections 3.1-3.3):
//   per expert e, tokens [cumsum[e], cumsum[e+1]):
//     gate_up = x @ w13_e (FP32),  sw = bf16(SiLU(gate) * up),  result = bf16(sw @ w2_e)
//
// Two launches of one persistent tcgen05 kind::f16 grouped GEMM:
//   GEMM1  A = prepared w13 tiles, 128 rows = 64 gate columns followed by the 64 up
//          columns of the same intermediate indices; B = token rows; the epilogue pairs
//          TMEM lanes r and 64 + r through shared memory and writes sw (bf16) to the
//          workspace.
//   GEMM2  A = prepared w2 tiles (128 output columns); B = rows of sw; the epilogue
//          rounds to bf16 and stores the result rows.
// As in the MXFP8 operator, weights are the 128-row operand (swap-AB), so an expert
// with few tokens streams each weight byte once; every CTA decodes the expert
// ranges itself; each (token group, column tile) unit covers the whole K range, so
// every output element is written once (no atomics, deterministic).
#include <cuda_bf16.h>

#include "common.cuh"
#include "pipeline.cuh"
#include "ptx.cuh"

namespace gmmfr {
namespace ffn {

constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kStageArena = 10 * 20480;  // 10 x 20480 (tmax 32), 8 x 24576 (64), 6 x 32768 (128)
constexpr int kMaxStages = 10;
constexpr int kOffX = kWTileBytes;  // token rows after the 16 KB weight tile
__host__ __device__ constexpr int stage_bytes(int tmax) { return kWTileBytes + tmax * 128; }
__host__ __device__ constexpr int n_stages(int tmax) { return tmax <= 32 ? 10 : (tmax <= 64 ? 8 : 6); }
static_assert(n_stages(32) * stage_bytes(32) <= kStageArena && n_stages(64) * stage_bytes(64) <= kStageArena &&
                  n_stages(128) * stage_bytes(128) <= kStageArena, "ring arena");
constexpr int kNumBars = 2 * kMaxStages + 6;
constexpr int kBarOff = kStageArena;
constexpr int kEndOff = kBarOff + kNumBars * 8;              // int32 s_end[1024]
constexpr int kGbaseOff = kEndOff + 4 * kMaxExperts;         // int32 s_gbase[1025]
constexpr int kScanOff = kGbaseOff + 4 * (kMaxExperts + 4);  // int64 scan scratch[8]
constexpr int kMiscOff = kScanOff + 8 * 8;                   // int32 misc[8]
constexpr int kXchgOff = kMiscOff + 32;                      // float [2][32][32]: up values for SwiGLU
constexpr int kSmemBytes = kXchgOff + 2 * 32 * 32 * 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr int kTmemCols = 256;  // two accumulators of up to 128 token columns

}  // namespace ffn

// ============================================================================ weight preparation
// GEMM1 tile (e, j, kb): row r < 64 holds gate column j*64 + r, row 64 + r the up column
// I + j*64 + r; 64 bf16 of K = H per row (k = kb*64 + c), 128-byte swizzled K-major
// image.  GEMM2 tile (e, j, kb): row r holds output column j*128 + r, K = I.  Padding is 0.
__global__ void __launch_bounds__(256) ffn_prep_kernel(FfnPrepParams p) {
  const int64_t t1 = (int64_t)p.E * p.NT1 * p.KB1;
  const int64_t t2 = (int64_t)p.E * p.NT2 * p.KB2;
  for (int64_t tile = blockIdx.x; tile < t1 + t2; tile += gridDim.x) {
    const bool first = tile < t1;
    const int64_t lt = first ? tile : tile - t1;
    const int KB = first ? p.KB1 : p.KB2, NT = first ? p.NT1 : p.NT2;
    const int64_t kb = lt % KB, j = (lt / KB) % NT, e = lt / ((int64_t)KB * NT);
    uint8_t* dst = p.prepared + tile * kWTileBytes;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int id = threadIdx.x + it * 256;
      const int r = id & 127, c = id >> 7;  // 16-byte chunk c of row r = 8 consecutive k
      int64_t col;
      bool col_ok;
      const uint16_t* src;
      int64_t ld, krows;
      if (first) {
        const int64_t i = j * 64 + (r & 63);
        col_ok = i < p.I;
        col = r < 64 ? i : p.I + i;
        src = p.w13 + e * p.H * (2 * p.I);  // w13_e [H, 2I]
        ld = 2 * p.I;
        krows = p.H;
      } else {
        col = j * 128 + r;
        col_ok = col < p.H;
        src = p.w2 + e * p.I * p.H;  // w2_e [I, H]
        ld = p.H;
        krows = p.I;
      }
      uint16_t v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int64_t k = kb * 64 + c * 8 + q;
        v[q] = (col_ok && k < krows) ? src[k * ld + col] : (uint16_t)0;
      }
      *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = *reinterpret_cast<const uint4*>(v);
    }
  }
}

cudaError_t launch_ffn_prep(const FfnPrepParams& p, cudaStream_t s) {
  const int64_t tiles = (int64_t)p.E * p.NT1 * p.KB1 + (int64_t)p.E * p.NT2 * p.KB2;
  if (tiles == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t grid = tiles < (int64_t)sms * 8 ? tiles : (int64_t)sms * 8;
  ffn_prep_kernel<<<(unsigned)grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ============================================================================ grouped GEMM
namespace {

struct FfnGroups {
  const int32_t* end;
  const int32_t* gbase;
  int E, tmax, start0;
  // e is also a hint (the expert of an earlier group of the range, or -1): walk forward from it
  __device__ void info(int g, int& e, int& t0, int& T) const {
    int lo;
    if (e >= 0 && gbase[e] <= g) {
      lo = e;
      while (gbase[lo + 1] <= g) ++lo;
    } else {
      lo = 0;
      int hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (gbase[mid] <= g) lo = mid; else hi = mid - 1;
      }
    }
    e = lo;
    const int start = lo ? end[lo - 1] : start0;
    t0 = start + (g - gbase[lo]) * tmax;
    const int rem = end[lo] - t0;
    T = rem < tmax ? rem : tmax;
  }
};

// Expert ranges from expert_cumsum: [start_e, end_e) with start_0 = clamp(cs[0], 0, N),
// start_e = end_{e-1}, end_e = clamp(cs[e+1], start_e, N); a cumsum that needs clamping
// sets kErrBadGroupList.  Chooses tmax and the first group of every expert.
__device__ int ffn_decode(const FfnParams& p, int32_t* s_end, int32_t* s_gbase, int64_t* scratch, uint32_t* s_err,
                          int& tmax_out, int& start0_out) {
  const int E = p.E;
  const int64_t N = p.N;
  const int tid = threadIdx.x;
  const int64_t c0 = p.cumsum[0];
  const int64_t start0 = c0 < 0 ? 0 : (c0 > N ? N : c0);
  if (tid == 0 && (c0 < 0 || c0 > N)) atomicOr(s_err, kErrBadGroupList);
  int64_t carry = start0;
  for (int base = 0; base < E; base += ffn::kThreads) {
    const int e = base + tid;
    const int64_t v = e < E ? p.cumsum[e + 1] : 0;
    const int64_t prev = e < E ? p.cumsum[e] : 0;
    if (e < E && (v < prev || v > N)) atomicOr(s_err, kErrBadGroupList);
    const int64_t c = e < E ? (v < 0 ? 0 : (v > N ? N : v)) : 0;
    int64_t tot;
    int64_t m = cta_scan<true, ffn::kThreads>(c, scratch, tot);
    m = m > carry ? m : carry;
    if (e < E) s_end[e] = (int32_t)m;
    carry = tot > carry ? tot : carry;
  }
  __syncthreads();
  int64_t mx = 0;
  for (int e = tid; e < E; e += ffn::kThreads) {
    const int64_t c = s_end[e] - (e ? s_end[e - 1] : start0);
    mx = c > mx ? c : mx;
  }
  int64_t mx_all;
  cta_scan<true, ffn::kThreads>(mx, scratch, mx_all);
  const int tmax = mx_all <= 32 ? 32 : (mx_all <= 64 ? 64 : 128);
  int64_t gcarry = 0;
  for (int base = 0; base < E; base += ffn::kThreads) {
    const int e = base + tid;
    const int64_t c = e < E ? s_end[e] - (e ? s_end[e - 1] : start0) : 0;
    const int64_t ng = (c + tmax - 1) / tmax;
    int64_t tot;
    const int64_t incl = cta_scan<false, ffn::kThreads>(ng, scratch, tot) + gcarry;
    if (e < E) s_gbase[e] = (int32_t)(incl - ng);
    gcarry += tot;
  }
  if (tid == 0) s_gbase[E] = (int32_t)gcarry;
  __syncthreads();
  tmax_out = tmax;
  start0_out = (int)start0;
  return (int)gcarry;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool epi_all(bool ok) {  // vote over the 4 epilogue warps
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u)
      : "memory");
  return r != 0;
}

}  // namespace

// kGateUp: GEMM1 with the SwiGLU epilogue (p.gate_up); a separate instantiation per GEMM keeps
// each launch's code to its own epilogue.
template <bool kGateUp>
__global__ void __launch_bounds__(ffn::kThreads, 1)
    ffn_gemm_kernel(const __grid_constant__ TokenMaps tmaps, const __grid_constant__ FfnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ffn::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + ffn::kMaxStages;
  uint64_t* accf = bars + 2 * ffn::kMaxStages;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  int32_t* s_end = reinterpret_cast<int32_t*>(smem + ffn::kEndOff);
  int32_t* s_gbase = reinterpret_cast<int32_t*>(smem + ffn::kGbaseOff);
  int64_t* s_scan = reinterpret_cast<int64_t*>(smem + ffn::kScanOff);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + ffn::kMiscOff);
  float* xchg = reinterpret_cast<float*>(smem + ffn::kXchgOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&misc[0]);
  int* abort_flag = &misc[1];
  uint32_t* s_err = reinterpret_cast<uint32_t*>(&misc[2]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if constexpr (kGateUp) ptx::griddep_launch_dependents();  // GEMM2 may launch (it waits for GEMM1 before reading sw)

  if (threadIdx.x == 0) {
    for (int s = 0; s < ffn::kMaxStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&accf[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&acce[b]), 4);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    *s_err = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane < 4) ptx::prefetch_tensormap(&tmaps.m[lane]);
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), ffn::kTmemCols);
    ptx::tmem_relinquish();
  }
  __syncthreads();
  int tmax, start0;
  const int n_groups = ffn_decode(p, s_end, s_gbase, s_scan, s_err, tmax, start0);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const FfnGroups groups{s_end, s_gbase, p.E, tmax, start0};
  const int stage_bytes = ffn::stage_bytes(tmax);
  const int n_stages = ffn::n_stages(tmax);
  const Ctl ctl{abort_flag, s_err, p.timeout_ns};
  // units (group, column tile), column tile fastest, in one contiguous range per CTA: a CTA
  // streams consecutive prepared tiles of one expert and re-reads that expert's token rows
  const int64_t n_units = (int64_t)n_groups * p.NT;
  const int64_t u_begin = n_units * blockIdx.x / gridDim.x, u_end = n_units * (blockIdx.x + 1) / gridDim.x;
  // (group, column tile) of the first unit; every role then steps the column tile, wrapping
  // into the next group, without dividing
  const int g_begin = (int)(u_begin / p.NT), j_begin = (int)(u_begin % p.NT);
  const uint32_t smem_base = ptx::smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_stream = ptx::l2_evict_first_policy();
      const uint64_t pol_keep = ptx::l2_evict_last_policy();
      int64_t n_fill = 0;  // stages filled; stage s was filled n_fill / n_stages (+1 if s < n_fill % n_stages) times
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // GEMM2 launched as a dependent of GEMM1: the weight tiles do not depend on GEMM1, so
      // the first ring's worth is requested before waiting for GEMM1 (the token rows, its
      // output, only after); those stages are remembered in `pend`
      bool waited = !p.dependent;
      int np = 0;
      int pend_stage[ffn::kMaxStages], pend_kb[ffn::kMaxStages], pend_t0[ffn::kMaxStages], pend_m[ffn::kMaxStages];
      auto token_rows = [&](uint32_t sb, uint32_t fb, int kb, int t0, int m) {
        int row = 0;  // a 128-row box, or a 64-row box, then 32-row boxes and a last 16-row box
        if (m == 8) {
          ptx::tma_load_2d(sb + ffn::kOffX, &tmaps.m[3], kb * 64, t0, fb, pol_keep);
          row = 128;
        } else if (m > 4) {
          ptx::tma_load_2d(sb + ffn::kOffX, &tmaps.m[2], kb * 64, t0, fb, pol_keep);
          row = 64;
        }
        for (; row < m * 16; row += 32) {
          const int last16 = row + 16 == m * 16;
          ptx::tma_load_2d(sb + ffn::kOffX + row * 128, &tmaps.m[last16 ? 0 : 1], kb * 64, t0 + row, fb, pol_keep);
        }
      };
      auto release_pending = [&]() {
        ptx::griddep_wait();
        for (int i = 0; i < np; ++i) {
          const uint32_t fb = ptx::smem_u32(&full[pend_stage[i]]);
          ptx::mbar_arrive_expect_tx(fb, pend_m[i] * 16 * 128);
          token_rows(smem_base + pend_stage[i] * stage_bytes, fb, pend_kb[i], pend_t0[i], pend_m[i]);
        }
        np = 0;
        waited = true;
      };
      int e = -1;
      for (int64_t u = u_begin, g = g_begin, j = j_begin; ok && u < u_end; ++u, j = (j + 1 == p.NT ? (++g, 0) : j + 1)) {
        int t0, T;
        groups.info((int)g, e, t0, T);
        const int m = (T + 15) / 16;
        const uint32_t tx = kWTileBytes + m * 16 * 128;
        const uint8_t* wsrc = p.prepared + ((int64_t)e * p.NT + j) * p.KB * (int64_t)kWTileBytes;
        const uint64_t pol_w = (s_gbase[e + 1] - s_gbase[e]) > 1 ? pol_keep : pol_stream;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!wait_bar(ptx::smem_u32(&empty[stage]), phase ^ 1, ctl)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full[stage]);
          const uint32_t sb = smem_base + stage * stage_bytes;
          if (waited) {
            ptx::mbar_arrive_expect_tx(fb, tx);
            ptx::bulk_g2s(sb, wsrc + (int64_t)kb * kWTileBytes, kWTileBytes, fb, pol_w);
            token_rows(sb, fb, kb, t0, m);
          } else {  // weights now; the arrival with the token rows after GEMM1
            ptx::mbar_expect_tx(fb, kWTileBytes);
            ptx::bulk_g2s(sb, wsrc + (int64_t)kb * kWTileBytes, kWTileBytes, fb, pol_w);
            pend_stage[np] = stage;
            pend_kb[np] = kb;
            pend_t0[np] = t0;
            pend_m[np] = m;
            if (++np == n_stages) release_pending();  // every stage is in use: the ring needs the tokens
          }
          ++n_fill;
          if (++stage == n_stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!waited) {
        if (ok) {
          release_pending();  // fewer items than stages
        } else {            // aborted: complete the pending phases without tokens so they can drain
          for (int i = 0; i < np; ++i) ptx::mbar_arrive(ptx::smem_u32(&full[pend_stage[i]]));
          np = 0;
          ptx::griddep_wait();
        }
      }
      if (ok) {
        for (int s = 0; s < n_stages; ++s) {
          const int64_t fs = n_fill / n_stages + (s < n_fill % n_stages ? 1 : 0);
          if (fs > 0 && !wait_bar(ptx::smem_u32(&empty[s]), (uint32_t)((fs - 1) & 1), ctl)) break;
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < n_stages; ++s) {
          const int64_t fs = n_fill / n_stages + (s < n_fill % n_stages ? 1 : 0);
          if (fs > 0) wait_bar_drain(ptx::smem_u32(&full[s]), (uint32_t)((fs - 1) & 1));
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      bool ok = true;
      int e = -1;
      for (int64_t u = u_begin, g = g_begin, j = j_begin; ok && u < u_end; ++u, j = (j + 1 == p.NT ? (++g, 0) : j + 1)) {
        int t0, T;
        groups.info((int)g, e, t0, T);
        const uint32_t npad = (uint32_t)((T + 15) / 16) * 16;
        const uint32_t idesc = p.idesc | ((npad >> 3) << 17);
        const int buf = acc_i & 1;
        if (!wait_bar(ptx::smem_u32(&acce[buf]), ((acc_i >> 1) & 1) ^ 1, ctl)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * tmax;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!wait_bar(ptx::smem_u32(&full[stage]), phase, ctl)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sb = smem_base + stage * stage_bytes;
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // K = 16 bf16 (32 bytes) per MMA
            const uint64_t adesc = ptx::smem_desc(sb + 32 * q, 16, 1024, ptx::kSwizzle128B);
            const uint64_t bdesc = ptx::smem_desc(sb + ffn::kOffX + 32 * q, 16, 1024, ptx::kSwizzle128B);
            ptx::tc_mma_f16(d_tmem, adesc, bdesc, idesc, (kb > 0 || q > 0) ? 1u : 0u);
          }
          ptx::tc_commit(ptx::smem_u32(&empty[stage]));
          if (++stage == n_stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        ptx::tc_commit(ptx::smem_u32(&accf[buf]));
        ++acc_i;
      }
      ptx::tc_commit(ptx::smem_u32(drain));
      wait_bar_drain(ptx::smem_u32(drain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int acc_i = 0;
    int e = -1;
    for (int64_t u = u_begin, g = g_begin, j = j_begin; u < u_end; ++u, j = (j + 1 == p.NT ? (++g, 0) : j + 1)) {
      int t0, T;
      groups.info((int)g, e, t0, T);
      const int buf = acc_i & 1;
      const bool ok = wait_bar(ptx::smem_u32(&accf[buf]), (acc_i >> 1) & 1, ctl);
      if (!epi_all(ok)) break;  // the 4 warps leave together: they share a named barrier
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * tmax;
      // 16 tokens per TMEM load: half the unrolled code of 32 (model shape 258.8 -> 256.4 us)
      for (int c0 = 0; c0 < T; c0 += 16) {
        uint32_t v[16];
        ptx::tmem_ld_32x32b_x16(taddr + c0, v);
        ptx::tmem_wait_ld();
        if (c0 + 16 >= T) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&acce[buf]));
        }
        const int cnt = T - c0 < 16 ? T - c0 : 16;
        if constexpr (kGateUp) {
          // lanes of quadrants 2, 3 hold the up columns matching quadrants 0, 1
          if (q >= 2) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) xchg[((q - 2) * 32 + jj) * 32 + lane] = __uint_as_float(v[jj]);
          }
          epi_bar();
          if (q < 2) {
            const int64_t col = (int64_t)j * 64 + q * 32 + lane;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              if (jj < cnt && col < p.out_cols) {
                const float gt = __uint_as_float(v[jj]);
                const float up = xchg[(q * 32 + jj) * 32 + lane];
                const float sw = gt / (1.0f + expf(-gt)) * up;
                p.out[((int64_t)t0 + c0 + jj) * p.out_cols + col] = __float2bfloat16_rn(sw);
              }
            }
          }
          epi_bar();
        } else {
          const int64_t col = (int64_t)j * kTileN + q * 32 + lane;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (jj < cnt && col < p.out_cols)
              p.out[((int64_t)t0 + c0 + jj) * p.out_cols + col] = __float2bfloat16_rn(__uint_as_float(v[jj]));
        }
      }
      ++acc_i;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, ffn::kTmemCols);
  }
  if (threadIdx.x == 0) {
    p.hdr[1 + p.slot_base + blockIdx.x] = *s_err;
    if (blockIdx.x == 0) p.hdr[0] = p.slot_base + gridDim.x;
  }
}

cudaError_t launch_ffn_gemm(const TokenMaps& tmaps, const FfnParams& p, int grid, cudaStream_t s) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(ffn_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, ffn::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ffn_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, ffn::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  auto kernel = p.gate_up ? ffn_gemm_kernel<true> : ffn_gemm_kernel<false>;
  if (!p.dependent) {
    kernel<<<grid, ffn::kThreads, ffn::kSmemBytes, s>>>(tmaps, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t lc = {};  // programmatic dependent of the previous kernel (GEMM1)
  lc.gridDim = dim3((unsigned)grid);
  lc.blockDim = dim3(ffn::kThreads);
  lc.dynamicSmemBytes = ffn::kSmemBytes;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, tmaps, p);
}

}  // namespace gmmfr

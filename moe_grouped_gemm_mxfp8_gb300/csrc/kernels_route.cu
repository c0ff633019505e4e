// MoE routing step before the operator: stable order of the flattened top-k
// expert ids, per-expert counts / prefix sums, and the token rows and their
// scales gathered into that order (LLaDA2.0-mini grouped-GEMM write-up,
// section 5.2: argsort, bincount, cumsum, gather).
//
// Entry f = b * topk + k has key id[f] when 0 <= id < E, else key E (routed
// nowhere, placed after every routed entry).  Output position of f:
//   base[key] + #{f' < f : key[f'] == key}
// computed in three launches:
//   route_count    per tile of 256 entries: in-tile stable rank of every entry
//                  and the tile's count per key
//   route_scan     one block: per-key totals, exclusive scan over keys, and the
//                  running per-key offset of every tile; group_list; error word
//   route_scatter  one warp per entry: perm, row_index, logit, the token row and
//                  its scale bytes copied to the entry's position
// Up to kFuseMaxM entries the three steps run as one launch (route_fused): every
// CTA reads all keys into shared memory (prefetching its slice's token rows into
// L2 meanwhile), counts them with shared-memory atomics (all entries, and those
// before its own slice), scans the counts, ranks its slice and scatters it.
// The redundant counting costs less than two extra launches at these sizes.
#include <cstdlib>

#include "common.cuh"
#include "ptx.cuh"

namespace gmmfr {

constexpr int kRouteTile = 256;
constexpr int kFuseMaxM = 8192;     // entries handled by the single-launch path
constexpr int kFuseThreads = 256;
constexpr int kFuseMaxSlice = 128;  // entries one CTA of that path ranks and scatters

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ int64_t load_id(const void* ids, int i32, int64_t f) {
  return i32 ? (int64_t) static_cast<const int32_t*>(ids)[f] : static_cast<const int64_t*>(ids)[f];
}

__global__ void __launch_bounds__(kRouteTile) route_count_kernel(RouteScatterParams p) {
  __shared__ int32_t s_cnt[kMaxExperts + 1];
  __shared__ int32_t s_key[kRouteTile / 32][32];
  __shared__ int32_t s_lead[kRouteTile / 32][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int keys = p.E + 1;
  for (int k = tid; k < keys; k += kRouteTile) s_cnt[k] = 0;
  const int64_t f = (int64_t)blockIdx.x * kRouteTile + tid;
  int key = -1;  // padding past M: a key of its own, never counted
  if (f < p.M) {
    const int64_t id = load_id(p.topk_ids, p.ids_i32, f);
    key = (id >= 0 && id < p.E) ? (int)id : p.E;
  }
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  const bool leader = lane == __ffs(peers) - 1;
  s_key[warp][lane] = key;
  s_lead[warp][lane] = leader ? __popc(peers) : 0;
  __syncthreads();
  int prefix = 0;  // entries with the same key in earlier warps of this tile
  for (int w = 0; w < warp; ++w)
#pragma unroll 8
    for (int l = 0; l < 32; ++l) prefix += s_key[w][l] == key ? s_lead[w][l] : 0;
  if (f < p.M) p.rank[f] = prefix + rank_w;
  if (leader && key >= 0) atomicAdd(&s_cnt[key], __popc(peers));
  __syncthreads();
  int32_t* tc = p.tile_counts + (int64_t)blockIdx.x * keys;
  for (int k = tid; k < keys; k += kRouteTile) tc[k] = s_cnt[k];
}

__global__ void __launch_bounds__(1024) route_scan_kernel(RouteScatterParams p) {
  __shared__ int64_t s_total[kMaxExperts + 1];
  __shared__ int64_t s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int keys = p.E + 1;
  const int64_t tiles = (p.M + kRouteTile - 1) / kRouteTile;
  for (int k = tid; k < keys; k += 1024) {
    int64_t t = 0;
    for (int64_t i = 0; i < tiles; ++i) t += p.tile_counts[i * keys + k];
    s_total[k] = t;
  }
  __syncthreads();
  // exclusive scan over keys (at most 1025: two rounds of 1024)
  int64_t carry = 0;
  for (int base = 0; base < keys; base += 1024) {
    const int k = base + tid;
    int64_t v = k < keys ? s_total[k] : 0;
    const int64_t orig = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int64_t w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t u = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += u;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int64_t incl = v + (warp > 0 ? s_warp[warp - 1] : 0);
    const int64_t total = s_warp[31];
    __syncthreads();
    if (k < keys) {
      const int64_t start = carry + incl - orig;  // first output position of key k
      if (k < p.E) p.group_list[k] = p.group_list_type == 1 ? orig : start + orig;
      int64_t running = start;  // each tile's first position for key k
      for (int64_t i = 0; i < tiles; ++i) {
        const int32_t c = p.tile_counts[i * keys + k];
        p.tile_counts[i * keys + k] = (int32_t)running;
        running += c;
      }
    }
    carry += total;
  }
  if (tid == 0) {
    p.hdr[0] = 1;
    p.hdr[1] = s_total[p.E] > 0 ? kErrBadExpertId : 0u;
  }
}

// n bytes from src to dst by one warp, eight independent loads in flight per lane.
__device__ __forceinline__ void copy_bytes(uint8_t* dst, const uint8_t* src, int64_t n, int lane) {
  for (int64_t i0 = lane; i0 < n; i0 += 32 * 8) {
    uint8_t r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (i0 + 32 * j < n) r[j] = __ldg(src + i0 + 32 * j);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (i0 + 32 * j < n) dst[i0 + 32 * j] = r[j];
  }
}

// Copies entry f (source row b = f / topk) to output position pos.
__device__ __forceinline__ void scatter_entry(const RouteScatterParams& p, int64_t f, int64_t pos, int lane) {
  const int64_t b = f / p.topk;
  if (lane == 0) {
    if (p.perm) p.perm[pos] = (int32_t)f;
    p.row_index[pos] = b;
    if (p.logit) p.logit[pos] = p.topk_weights ? p.topk_weights[f] : 1.f;
  }
  const uint8_t* src = p.x + b * p.K;
  uint8_t* dst = p.x1 + pos * p.K;
  if (p.vec16) {  // 8 independent 16-byte loads in flight per lane, then their stores
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const int64_t n16 = p.K / 16;
    for (int64_t i0 = lane; i0 < n16; i0 += 32 * 8) {
      uint4 r[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (i0 + 32 * j < n16) r[j] = __ldg(s4 + i0 + 32 * j);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (i0 + 32 * j < n16) d4[i0 + 32 * j] = r[j];
    }
  } else {
    copy_bytes(dst, src, p.K, lane);
  }
  const int64_t sb = 2 * (int64_t)p.Ks;
  copy_bytes(p.pertoken_scale + pos * sb, p.x_scale + b * sb, sb, lane);
}

__global__ void __launch_bounds__(256) route_scatter_kernel(RouteScatterParams p) {
  ptx::griddep_launch_dependents();  // the operator that follows may start launching (it waits for us)
  const int lane = threadIdx.x & 31;
  const int64_t f = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (f >= p.M) return;
  const int64_t id = load_id(p.topk_ids, p.ids_i32, f);
  const int key = (id >= 0 && id < p.E) ? (int)id : p.E;
  scatter_entry(p, f, (int64_t)p.tile_counts[(f / kRouteTile) * (p.E + 1) + key] + p.rank[f], lane);
}

__global__ void __launch_bounds__(kFuseThreads, 3) route_fused_kernel(RouteScatterParams p) {
  __shared__ int32_t s_key[kFuseMaxM];
  __shared__ int32_t s_cnt[kMaxExperts + 1];   // entries per key
  __shared__ int32_t s_base[kMaxExperts + 1];  // first output position of each key
  __shared__ int32_t s_run[kMaxExperts + 1];   // per key: entries before the next one to rank
  __shared__ int32_t s_pos[kFuseMaxSlice];
  __shared__ int32_t s_wsum[kFuseThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  ptx::griddep_launch_dependents();  // the operator that follows may start launching (it waits for us)
  const int keys = p.E + 1;
  const int M = (int)p.M;
  const int f_lo = (int)((int64_t)M * blockIdx.x / gridDim.x);
  const int f_hi = (int)((int64_t)M * (blockIdx.x + 1) / gridDim.x);
  for (int k = tid; k < keys; k += kFuseThreads) {
    s_cnt[k] = 0;
    s_run[k] = 0;
  }
  // keys of all entries into shared memory, eight independent loads in flight per thread
  for (int base = 0; base < M; base += 8 * kFuseThreads) {
    int64_t id[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int f = base + j * kFuseThreads + tid;
      id[j] = f < M ? load_id(p.topk_ids, p.ids_i32, f) : 0;
    }
    // the slice's source rows are known before their positions (entry f reads token f / topk):
    // pull them and their scales into L2 while the keys are loaded, counted and scanned
    if (base == 0) {
      for (int i = warp; i < f_hi - f_lo; i += kFuseThreads / 32) {
        const int64_t b = (f_lo + i) / p.topk;
        const int64_t sb = 2 * (int64_t)p.Ks;
        for (int64_t o = (int64_t)lane * 128; o < p.K; o += 32 * 128) prefetch_l2(p.x + b * p.K + o);
        for (int64_t o = (int64_t)lane * 128; o < sb; o += 32 * 128) prefetch_l2(p.x_scale + b * sb + o);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int f = base + j * kFuseThreads + tid;
      if (f < M) s_key[f] = (id[j] >= 0 && id[j] < p.E) ? (int)id[j] : p.E;
    }
  }
  __syncthreads();
  // per key: all entries, and those before this CTA's slice.  Shared-memory atomics, one per
  // entry; a warp whose 32 keys are equal adds them in one.  (Grouping equal keys with
  // __match_any_sync first cost ~0.75 us per 256 entries at 256 experts, as its time grows with
  // the number of distinct keys in the warp: 12 of the 22 us of a 4096-entry launch.)
  for (int base = 0; base < M; base += kFuseThreads) {  // uniform trip count (warp-wide votes)
    const int f = base + tid;
    const int key = f < M ? s_key[f] : -1;
    if (__reduce_min_sync(0xffffffffu, key) == __reduce_max_sync(0xffffffffu, key)) {
      const unsigned before = __ballot_sync(0xffffffffu, f < f_lo);
      if (lane == 0 && key >= 0) {
        atomicAdd(&s_cnt[key], 32);
        if (before) atomicAdd(&s_run[key], __popc(before));
      }
    } else {
      if (key >= 0) atomicAdd(&s_cnt[key], 1);
      if (f < f_lo) atomicAdd(&s_run[key], 1);
    }
  }
  __syncthreads();
  // exclusive scan of the counts over keys: each thread sums a run of consecutive keys
  constexpr int kPer = (kMaxExperts + 1 + kFuseThreads - 1) / kFuseThreads;
  const int k0 = tid * kPer;
  int local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) local += (k0 + i < keys) ? s_cnt[k0 + i] : 0;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += s_wsum[w];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    if (k0 + i < keys) {
      s_base[k0 + i] = run;
      run += s_cnt[k0 + i];
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int k = tid; k < p.E; k += kFuseThreads)
      p.group_list[k] = p.group_list_type == 1 ? (int64_t)s_cnt[k] : (int64_t)(s_base[k] + s_cnt[k]);
    if (tid == 0) {
      p.hdr[0] = 1;
      p.hdr[1] = s_cnt[p.E] > 0 ? kErrBadExpertId : 0u;
    }
  }
  // positions of this CTA's slice, 32 entries at a time in entry order (warp 0)
  if (warp == 0) {
    for (int c = f_lo; c < f_hi; c += 32) {
      const int f = c + lane;
      const int key = f < f_hi ? s_key[f] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      if (f < f_hi) s_pos[f - f_lo] = s_base[key] + s_run[key] + __popc(peers & ((1u << lane) - 1u));
      __syncwarp();
      if (key >= 0 && lane == __ffs(peers) - 1) s_run[key] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int i = warp; i < f_hi - f_lo; i += kFuseThreads / 32) scatter_entry(p, f_lo + i, s_pos[i], lane);
}

cudaError_t launch_route_kernels(const RouteScatterParams& p, cudaStream_t s) {
  const bool split_only = std::getenv("GMMFR_ROUTE_SPLIT") != nullptr;  // testing aid: force 3 launches
  if (p.M <= kFuseMaxM && !split_only) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t grid = (p.M + 7) / 8;  // about one entry per warp
    if (grid > 3 * sms) grid = 3 * sms;  // one wave: three CTAs per SM (77 registers, no spills)
    const int64_t min_grid = (p.M + kFuseMaxSlice - 1) / kFuseMaxSlice;  // every slice fits s_pos
    if (grid < min_grid) grid = min_grid;
    if (grid < 1) grid = 1;
    route_fused_kernel<<<(unsigned)grid, kFuseThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  const int64_t tiles = (p.M + kRouteTile - 1) / kRouteTile;
  if (tiles > 0) {
    route_count_kernel<<<(unsigned)tiles, kRouteTile, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  route_scan_kernel<<<1, 1024, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.M == 0) return e;
  route_scatter_kernel<<<(unsigned)((p.M + 7) / 8), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gmmfr

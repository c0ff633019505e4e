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
#include "common.cuh"

namespace gmmfr {

constexpr int kRouteTile = 256;

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

__global__ void __launch_bounds__(256) route_scatter_kernel(RouteScatterParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t f = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (f >= p.M) return;
  const int64_t id = load_id(p.topk_ids, p.ids_i32, f);
  const int key = (id >= 0 && id < p.E) ? (int)id : p.E;
  const int64_t pos = (int64_t)p.tile_counts[(f / kRouteTile) * (p.E + 1) + key] + p.rank[f];
  const int64_t b = f / p.topk;
  if (lane == 0) {
    if (p.perm) p.perm[pos] = (int32_t)f;
    p.row_index[pos] = b;
    if (p.logit) p.logit[pos] = p.topk_weights ? p.topk_weights[f] : 1.f;
  }
  const uint8_t* src = p.x + b * p.K;
  uint8_t* dst = p.x1 + pos * p.K;
  if (p.vec16) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int64_t i = lane; i < p.K / 16; i += 32) d4[i] = s4[i];
  } else {
    for (int64_t i = lane; i < p.K; i += 32) dst[i] = src[i];
  }
  const int64_t sb = 2 * (int64_t)p.Ks;
  for (int64_t i = lane; i < sb; i += 32) p.pertoken_scale[pos * sb + i] = p.x_scale[b * sb + i];
}

cudaError_t launch_route_kernels(const RouteScatterParams& p, cudaStream_t s) {
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

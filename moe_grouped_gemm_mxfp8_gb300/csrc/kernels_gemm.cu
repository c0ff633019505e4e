// Persistent grouped GEMM of MXFP8 grouped-matmul-finalize-routing on sm_103a.
//
// Work: for every token group g (at most `tmax` routed tokens of one expert e),
// every 128-column tile j of the output and every K block kb of 128 bytes per row,
//   D[n, t] += sum_{k in block} (x2[e,k,n] * s_w) * (x1[t,k] * s_x)
// with tcgen05.mma kind::mxf8f6f4 block_scale (FP8: 128 K elements per block), or
// kind::mxf4 block_scale when tokens and weights are both packed E2M1 (256 K elements
// per block, two per byte); one E8M0 scale per 32 K elements either way.
// The weights are the 128-row A operand (rows = output columns), the tokens the
// N-wide B operand (N = tokens rounded up to 16), so experts holding few tokens
// still stream each weight byte exactly once.
//
// Every CTA first decodes group_list itself (at most 1024 experts) into shared
// memory: contiguous expert ranges, the token group width tmax in {32, 64, 128}
// (the smallest that holds the largest expert, so a skewed routing re-reads as
// few weight tiles as possible), and the first group of every expert.  The
// shared-memory ring is then cut into as many stages as fit for that width.
//
// Roles (224 threads for FP8 operands, 256 for packed E2M1; one CTA per SM):
//   warp 0     TMA producer: prepared weight tile + its scales (one bulk copy) and
//              the token rows (boxes of 128, 64, 32 or 16 rows)
//   warp 1     TMEM owner and MMA issuer (scale copies to TMEM, 4 MMAs per stage)
//   warps 2-5  epilogue: TMEM -> registers, + bias, x logit, red.global.add.f32 into
//              out[row_index[t], n] (or a plain store into the per-token buffer in
//              deterministic mode); before the first tile they add the shared
//              input for their slice of rows.
//   warp 6     token-scale packer: pertoken_scale bytes of the stage's tokens into the
//              32-row x 16-byte layout tcgen05.cp spreads over TMEM lanes; with packed
//              E2M1 warps 6 and 7 take the even and odd stages.
//
// Scheduling: atomic mode splits the total (group, tile, K-block) iteration space
// over the CTAs in contiguous ranges (stream-K) of equal item count, or, when token
// groups of 64 or 128 are in play, of equal cost (item_cost: CTAs holding 128-token
// groups get fewer items than those holding 16-token ones); a tile cut between CTAs is finished by
// atomics, which is exact up to FP32 rounding order since every term is linear.
// Deterministic mode gives each (group, tile, K-split) unit to one CTA (contiguous
// ranges of units) and stores its result for the row-ordered combine.
//
// Every wait is bounded: on timeout the CTA sets GMMFR_DEV_TIMEOUT, stops
// issuing, waits (bounded) for its copies and MMAs in flight, frees TMEM and exits.
#include "common.cuh"
#include "pipeline.cuh"
#include "ptx.cuh"

namespace gmmfr {

namespace cfg {
// One ring of stages; a stage holds everything one K block of a segment needs:
//   [0, 16384)        weight tile, 128 rows x 128 bytes (1024-aligned, 128-byte swizzle)
//   [16384, +S)       its E8M0 scales (same bulk copy); S = 512 (FP8: 4 per row) or
//                     1024 (packed E2M1: 8 per row, two 512-byte chunks)
//   [16384 + S, +S)   the token scales (packed by warp 6), same layout
//   [16384 + 2S, ...) tmax token rows of 128 bytes (1024-aligned, 128-byte swizzle)
// Loaded L2 latency is about that of HBM here, so token rows need the same lead
// time as weights and share the stage.
constexpr int kMaxStages = 10;
constexpr int kOffWSF = kWTileBytes;
__host__ __device__ constexpr int sf_bytes(bool fp4) { return fp4 ? 2 * kSfChunk : kSfChunk; }
__host__ __device__ constexpr int off_xsf(bool fp4) { return kWTileBytes + sf_bytes(fp4); }
__host__ __device__ constexpr int off_x(bool fp4) { return kWTileBytes + 2 * sf_bytes(fp4); }
__host__ __device__ constexpr int stage_bytes(int tmax, bool fp4) { return off_x(fp4) + tmax * 128; }
__host__ __device__ constexpr int n_stages(int tmax, bool fp4) {
  return tmax <= 32 ? (fp4 ? 9 : 10) : (tmax <= 64 ? 8 : 6);
}
// FP8: 10 x 21504 (tmax 32), 8 x 25600 (64), 6 x 33792 (128);
// E2M1: 9 x 22528, 8 x 26624, 6 x 34816
constexpr int kArena = 10 * 21504;
static_assert(n_stages(32, false) * stage_bytes(32, false) <= kArena &&
                  n_stages(64, false) * stage_bytes(64, false) <= kArena &&
                  n_stages(128, false) * stage_bytes(128, false) <= kArena &&
                  n_stages(32, true) * stage_bytes(32, true) <= kArena &&
                  n_stages(64, true) * stage_bytes(64, true) <= kArena &&
                  n_stages(128, true) * stage_bytes(128, true) <= kArena,
              "ring arena");
static_assert(off_x(true) % 1024 == 0 && stage_bytes(32, true) % 1024 == 0 && off_x(false) % 1024 == 0 &&
                  stage_bytes(32, false) % 1024 == 0,
              "swizzled operands need 1024-byte alignment");
__host__ __device__ constexpr int sf_cols(bool fp4) { return fp4 ? 16 : 8; }  // TMEM scale columns per stage
constexpr int kTmemCols = 512;  // 2 x tmax accumulator columns + the scale columns of every stage
static_assert(2 * 128 + sf_cols(true) * n_stages(128, true) <= kTmemCols &&
                  2 * 64 + sf_cols(true) * n_stages(64, true) <= kTmemCols &&
                  2 * 32 + sf_cols(true) * n_stages(32, true) <= kTmemCols &&
                  2 * 128 + sf_cols(false) * n_stages(128, false) <= kTmemCols &&
                  2 * 64 + sf_cols(false) * n_stages(64, false) <= kTmemCols &&
                  2 * 32 + sf_cols(false) * n_stages(32, false) <= kTmemCols,
              "TMEM");
constexpr int kNumBars = 2 * kMaxStages + 6;
constexpr int kBarOff = kArena;
constexpr int kEndOff = kBarOff + kNumBars * 8;              // int32 s_end[1024]
constexpr int kGbaseOff = kEndOff + 4 * kMaxExperts;         // int32 s_gbase[1025]
constexpr int kWbaseOff = kGbaseOff + 4 * (kMaxExperts + 4); // int32 s_wbase[1025]
constexpr int kScanOff = kWbaseOff + 4 * (kMaxExperts + 4);  // int64 scan scratch[8]
static_assert(gemm_threads(true) <= 8 * 32 && gemm_threads(false) <= 8 * 32, "scan scratch: one word per warp");
constexpr int kMiscOff = kScanOff + 8 * 8;                   // int32 misc[8]
constexpr int kTokOff = kMiscOff + 32;                       // int32 rows[2][128], float logits[2][128]
constexpr int kSmemBytes = kTokOff + 2 * 2 * 128 * 4 + 1024; // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
}  // namespace cfg

struct Seg {
  int g, j, kb0, kb1, slot;
};

// Relative time of one (group, tile, K block) item of a group of T tokens: the prepared
// weight tile with its scales (132 units of 128 bytes, from HBM) weighted 3:1 against the
// token rows (16 at a time, mostly L2 hits, re-read by every column tile) — the ratio that
// evened out per-CTA finish times on a Zipf routing with 1 to 128 tokens per group.
__host__ __device__ constexpr int item_cost(int T) { return 3 * (kPrepTileBytes / 128) + 16 * ((T + 15) / 16); }

// Expert ranges and token groups decoded from group_list, in shared memory.
struct Groups {
  const int32_t* end;    // end of expert e's token range (ranges are contiguous from 0)
  const int32_t* gbase;  // first group of expert e; gbase[E] = number of groups
  const int32_t* wbase;  // cost of the items of experts before e in one K block of one tile
                         // (item_cost units); wbase[E] = total, < 0 when it would overflow
  int E, tmax;
  // group g -> expert, first token, tokens.  e is also a hint: the expert of an earlier
  // group of the same range (or -1); the walk forward from it replaces the binary search
  // when g has not wrapped below it.
  __device__ void info(int g, int& e, int& t0, int& T) const {
    int lo;  // largest e with gbase[e] <= g (always a non-empty expert)
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
    const int start = lo ? end[lo - 1] : 0;
    const int i = g - gbase[lo];
    t0 = start + i * tmax;
    const int rem = end[lo] - t0;
    T = rem < tmax ? rem : tmax;
  }
  // First item (index tile * KB + kb, tile = j * n_groups + g) whose cost prefix reaches x.
  __device__ int64_t item_at(int64_t x, int KB, int NT, int n_groups) const {
    const int64_t row = (int64_t)KB * wbase[E];  // all items of one column tile
    const int64_t j = x / row;
    if (j >= NT) return (int64_t)n_groups * NT * KB;
    const int64_t r = x - j * row;
    int lo = 0, hi = E - 1;  // the last expert whose items start at or before r (it holds tokens)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)KB * wbase[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int ng = gbase[e + 1] - gbase[e];
    const int64_t wf = item_cost(tmax);
    const int64_t re = r - (int64_t)KB * wbase[e];
    int64_t gl = re / ((int64_t)KB * wf);
    if (gl > ng - 1) gl = ng - 1;
    const int last_t = end[e] - (e ? end[e - 1] : 0) - (ng - 1) * tmax;
    const int64_t wg = gl < ng - 1 ? wf : item_cost(last_t);
    const int64_t rg = re - gl * KB * wf;
    return (j * n_groups + gbase[e] + gl) * KB + (rg + wg - 1) / wg;  // kb == KB is the next tile
  }
};

// The sequence of (group, tile, K range) segments of one CTA; every role walks it.
// With the even split (token groups of at most 32) the atomic mode orders the items
// group-major (tile = g * NT + j): a CTA's range then reads an expert's prepared tiles in
// address order, the order bulk copies stream fastest in, and keeps each group's token rows
// for all its column tiles (C5 1086 -> 1076 us against column-tile-major order); deterministic
// mode's units (tile, then K split) follow the same order when every expert is one group.
// With the cost-weighted split, or token groups wider than 32 in deterministic mode, tiles
// stay column-tile-major (tile = j * n_groups + g), so the groups of one expert that holds more
// than tmax tokens are adjacent and re-read their shared weight tiles while still in L2
// (group-major cost C4 11 us).  The walk steps (major, minor) = (g, j) or (j, g) with selects,
// not branches.
struct Sched {
  int64_t i, i_end, step;
  int NT, KB, split, ng;
  bool det;
  bool gmajor;               // atomic mode, even split: tile = g * NT + j
  // item i's K block (deterministic mode: K split) and tile: cur_g = the major and cur_j = the
  // minor tile index (group and column tile, or column tile and group)
  int cur_g, cur_j, cur_kb;
  __device__ void init(int n_groups, int NT_, int KB_, bool det_, int split_, bool reverse, const Groups& gr) {
    ng = n_groups;
    NT = NT_;
    KB = KB_;
    det = det_;
    split = split_;
    const int64_t tiles = (int64_t)n_groups * NT;
    if (det) {
      // contiguous ranges of (group, tile, K split) units: unit u = tile * split + sp, walked
      // from the first without dividing (cur_kb holds sp), or from the last when `reverse`
      // (every unit writes its own slice of the per-token buffer, so the order in which a CTA
      // takes its units cannot change the result; tests walk both ways)
      const int64_t units = tiles * split;
      i = units * blockIdx.x / gridDim.x;
      i_end = units * (blockIdx.x + 1) / gridDim.x;
      step = reverse ? -1 : 1;
      const int64_t first = reverse && i_end > i ? i_end - 1 : i;
      const int64_t tile = first / split;
      cur_kb = (int)(first - tile * split);
      gmajor = gr.tmax <= 32;  // one token group per expert: group-major, as in atomic mode
      const int64_t minors = gmajor ? NT : (ng > 0 ? ng : 1);
      cur_g = (int)(tile / minors);
      cur_j = (int)(tile - cur_g * minors);
      return;
    }
    step = 0;
    gmajor = gr.wbase[gr.E] <= 0;
    if (!gmajor) {
      // equal cost per CTA: items of large token groups move more bytes than those of small ones
      const int64_t total = (int64_t)NT * KB * gr.wbase[gr.E];
      i = gr.item_at(total * blockIdx.x / gridDim.x, KB, NT, n_groups);
      i_end = gr.item_at(total * (blockIdx.x + 1) / gridDim.x, KB, NT, n_groups);
    } else {
      const int64_t total = tiles * KB;
      if (total * gridDim.x < ((int64_t)1 << 32)) {  // 32-bit division where it fits
        i = (uint32_t)(total * blockIdx.x) / gridDim.x;
        i_end = (uint32_t)(total * (blockIdx.x + 1)) / gridDim.x;
      } else {
        i = total * blockIdx.x / gridDim.x;
        i_end = total * (blockIdx.x + 1) / gridDim.x;
      }
    }
    // position of the first item (tile = major * minors + minor); next() then walks tiles
    // without dividing.  cur_g holds the major index, cur_j the minor one.
    const int64_t tile = i / KB;
    cur_kb = (int)(i - tile * KB);
    const int64_t minors = gmajor ? NT : (ng > 0 ? ng : 1);
    cur_g = (int)(tile / minors);
    cur_j = (int)(tile - cur_g * minors);
  }
  // kDet: the kernel's mode (compile time, so each instantiation holds one walk)
  template <bool kDet>
  __device__ __forceinline__ bool next(Seg& s) {
    if (i >= i_end) return false;
    if constexpr (!kDet) {  // tiles in (major, minor) order; a segment runs to its tile's end or the range's
      s.g = gmajor ? cur_g : cur_j;
      s.j = gmajor ? cur_j : cur_g;
      s.kb0 = cur_kb;
      const int64_t left = i_end - i;
      s.kb1 = (KB - cur_kb) < left ? KB : cur_kb + (int)left;
      s.slot = 0;
      i += s.kb1 - s.kb0;
      cur_kb = 0;
      if (++cur_j == (gmajor ? NT : ng)) {
        cur_j = 0;
        ++cur_g;
      }
      return true;
    } else {  // deterministic: the next (group, tile, K split) unit of this CTA's range
      const int sp = cur_kb;
      s.g = gmajor ? cur_g : cur_j;
      s.j = gmajor ? cur_j : cur_g;
      s.kb0 = (int)((int64_t)sp * KB / split);
      s.kb1 = (int)((int64_t)(sp + 1) * KB / split);
      s.slot = sp;
      ++i;
      const int minors = gmajor ? NT : ng;
      if (step > 0) {
        if (++cur_kb == split) {
          cur_kb = 0;
          if (++cur_j == minors) {
            cur_j = 0;
            ++cur_g;
          }
        }
      } else if (--cur_kb < 0) {
        cur_kb = split - 1;
        if (--cur_j < 0) {
          cur_j = minors - 1;
          --cur_g;
        }
      }
      return true;
    }
  }
};

__device__ __forceinline__ int load_row32(const void* rows, int row_i32, int64_t t, int64_t batch) {
  const int64_t r = row_i32 ? (int64_t) static_cast<const int32_t*>(rows)[t] : static_cast<const int64_t*>(rows)[t];
  return (r >= 0 && r < batch) ? (int)r : -1;
}

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Expert ranges (MXFP8 grouped_matmul_finalize_routing write-up, section 4.3:
// type 0 prefix sums, type 1 counts),
// made contiguous and clamped to [0, M]; sets kErrBadGroupList when clamping was
// needed.  Fills s_end, chooses tmax, fills s_gbase.  Returns the group count.
// g0 = group_list[threadIdx.x] (0 past E), loaded by the caller at kernel entry so that
// its latency overlaps the barrier and TMEM set-up.
template <int kThreads>
__device__ int decode_groups(const GemmParams& p, int64_t g0, int32_t* s_end, int32_t* s_gbase, int32_t* s_wbase,
                             int64_t* scratch, uint32_t* s_err, int& tmax_out) {
  const int E = p.E;
  const int64_t M = p.M;
  const int tid = threadIdx.x;
  int64_t carry = 0;
  for (int base = 0; base < E; base += kThreads) {  // uniform trip count
    const int e = base + tid;
    const int64_t g = base == 0 ? g0 : (e < E ? p.group_list[e] : 0);
    int64_t v, tot;
    if (p.group_list_type == 1) {
      if (e < E && g < 0) atomicOr(s_err, kErrBadGroupList);
      const int64_t c = e < E ? (g < 0 ? 0 : (g > M ? M + 1 : g)) : 0;
      v = cta_scan<false, kThreads>(c, scratch, tot) + carry;
      carry += tot;
    } else {
      const int64_t prev = (e > 0 && e < E) ? p.group_list[e - 1] : 0;
      if (e < E && (g < prev || g > M)) atomicOr(s_err, kErrBadGroupList);
      const int64_t c = e < E ? (g < 0 ? 0 : (g > M ? M : g)) : 0;
      v = cta_scan<true, kThreads>(c, scratch, tot);
      v = v > carry ? v : carry;
      carry = tot > carry ? tot : carry;
    }
    if (e < E) s_end[e] = (int32_t)(v < M ? v : M);
  }
  if (p.group_list_type == 1 && tid == 0 && carry > M) atomicOr(s_err, kErrBadGroupList);
  __syncthreads();
  // largest expert -> token group width
  int64_t mx = 0;
  for (int e = tid; e < E; e += kThreads) {
    const int64_t c = s_end[e] - (e ? s_end[e - 1] : 0);
    mx = c > mx ? c : mx;
  }
  int64_t mx_all;
  cta_scan<true, kThreads>(mx, scratch, mx_all);
  int tmax = mx_all <= 32 ? 32 : (mx_all <= 64 ? 64 : 128);
  if (p.tmax_fixed) tmax = p.tmax_fixed;
  // first group of every expert, and (when groups can differ much in size) the cost prefix
  // of the experts' items
  const bool weigh = tmax >= 64;
  int64_t gcarry = 0, wcarry = 0;
  for (int base = 0; base < E; base += kThreads) {
    const int e = base + tid;
    const int64_t c = e < E ? s_end[e] - (e ? s_end[e - 1] : 0) : 0;
    const int64_t ng = (c + tmax - 1) / tmax;
    const int64_t w = ng > 0 ? (ng - 1) * item_cost(tmax) + item_cost((int)(c - (ng - 1) * tmax)) : 0;
    int64_t tot, wtot;
    const int64_t incl = cta_scan<false, kThreads>(ng, scratch, tot) + gcarry;
    int64_t wincl = 0;
    wtot = 0;
    if (weigh) wincl = cta_scan<false, kThreads>(w, scratch, wtot) + wcarry;  // uniform branch
    if (e < E) {
      s_gbase[e] = (int32_t)(incl - ng);
      s_wbase[e] = (int32_t)((wincl - w) < INT32_MAX ? wincl - w : INT32_MAX);
    }
    gcarry += tot;
    wcarry += wtot;
  }
  if (tid == 0) {
    s_gbase[E] = (int32_t)gcarry;
    s_wbase[E] = weigh && wcarry < INT32_MAX ? (int32_t)wcarry : -1;  // -1: split by item count instead
  }
  __syncthreads();
  tmax_out = tmax;
  return (int)gcarry;
}

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

// Deterministic mode: the tokens of each out row (CSR, unordered within a row; the combine
// orders them), from the covered tokens [0, covered) of the decoded expert ranges.  Built by
// the 128 epilogue threads of one CTA (named barrier 1) before its first tile, in time those
// warps spend waiting anyway; the combine kernel reads it after this kernel has completed.
__device__ void build_row_csr(const GemmParams& p, int64_t covered, int ep_tid, int64_t* scratch) {
  const int lane = ep_tid & 31, w = ep_tid >> 5;
  for (int64_t r = ep_tid; r < p.batch; r += 128) p.csr_cnt[r] = 0;
  __threadfence_block();
  ptx::bar_sync(1, 128);
  for (int64_t t = ep_tid; t < covered; t += 128) {
    const int r = load_row32(p.row_index, p.row_i32, t, p.batch);
    if (r >= 0) atomicAdd(&p.csr_cnt[r], 1);
  }
  __threadfence_block();
  ptx::bar_sync(1, 128);
  int64_t running = 0;  // exclusive scan of the counts, 128 rows at a time
  for (int64_t base = 0; base < p.batch; base += 128) {
    const int64_t r = base + ep_tid;
    const int c = r < p.batch ? __ldcg(&p.csr_cnt[r]) : 0;  // counts were made by atomics (L2)
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) scratch[w] = incl;
    ptx::bar_sync(1, 128);
    int64_t before = 0, chunk = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t v = scratch[k];
      before += k < w ? v : 0;
      chunk += v;
    }
    if (r < p.batch) {
      const int32_t start = (int32_t)(running + before + incl - c);
      p.csr_row_ptr[r] = start;
      p.csr_cursor[r] = start;
    }
    running += chunk;
    ptx::bar_sync(1, 128);  // scratch is rewritten by the next chunk
  }
  if (ep_tid == 0) p.csr_row_ptr[p.batch] = (int32_t)running;
  __threadfence_block();
  ptx::bar_sync(1, 128);
  for (int64_t t = ep_tid; t < covered; t += 128) {
    const int r = load_row32(p.row_index, p.row_i32, t, p.batch);
    if (r >= 0) p.csr_sorted[atomicAdd(&p.csr_cursor[r], 1)] = (int32_t)t;
  }
}

// The four E8M0 bytes of token t for the 32-element blocks 4*c .. 4*c+3 (c = kb for FP8
// blocks, 2*kb and 2*kb + 1 for the two halves of a packed E2M1 block); blocks starting at
// or past K are padding: 127 = 1.0.
__device__ __forceinline__ bool scale_words_aligned(const GemmParams& p) {
  return ((reinterpret_cast<uintptr_t>(p.pertoken_scale) | (uintptr_t)(2 * p.Ks)) & 3) == 0;
}
__device__ __forceinline__ uint32_t token_scale_word(const GemmParams& p, int64_t t, int c) {
  const uint8_t* src = p.pertoken_scale + t * 2 * (int64_t)p.Ks + 4 * c;
  if (scale_words_aligned(p) && (int64_t)(4 * c + 3) * 32 < p.K) return *reinterpret_cast<const uint32_t*>(src);
  uint32_t w = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) w |= ((int64_t)(4 * c + q) * 32 < p.K ? (uint32_t)src[q] : 127u) << (8 * q);
  return w;
}

// Item iterator of the token-scale packer: one (segment, K block) per stage.
struct PackIter {
  Seg sg;
  int kb, kb1, t0, T;
  int e;  // expert of the current segment (hint for the next lookup)
  bool valid;
};

template <bool kDet>
__device__ __forceinline__ bool pack_next(PackIter& it, Sched& sched, const Groups& groups) {
  if (it.valid && ++it.kb < it.kb1) return true;
  while (sched.next<kDet>(it.sg)) {
    groups.info(it.sg.g, it.e, it.t0, it.T);
    it.kb = it.sg.kb0;
    it.kb1 = it.sg.kb1;
    if (it.kb < it.kb1) {
      it.valid = true;
      return true;
    }
  }
  it.valid = false;
  return false;
}

// Scale words of tokens lane, lane+32, lane+64, lane+96 of the item (127 = 1.0 past the
// group): w[r] for the item's 32-blocks 0..3, and with packed E2M1 w[4 + r] for 4..7.
template <bool fp4>
__device__ __forceinline__ void pack_load(const GemmParams& p, const PackIter& it, uint32_t (&w)[8]) {
  const int lane = threadIdx.x & 31;
  const int c = fp4 ? 2 * it.kb : it.kb;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = lane + 32 * r;
    const bool in = it.valid && i < it.T;
    w[r] = in ? token_scale_word(p, (int64_t)it.t0 + i, c) : 0x7F7F7F7Fu;
    w[4 + r] = (fp4 && in) ? token_scale_word(p, (int64_t)it.t0 + i, c + 1) : 0x7F7F7F7Fu;
  }
}

// fp4: packed E2M1 operands (kind::mxf4); det: deterministic mode.  Separate instantiations
// keep each variant's loops free of the others' code (the instruction cache is the scarce
// resource: one in five fetches misses it).
template <bool fp4, bool det>
__global__ void __launch_bounds__(gemm_threads(fp4), 1)
    gemm_kernel(const __grid_constant__ TokenMaps tmaps, const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + cfg::kBarOff);
  uint64_t* full = bars;                         // [kMaxStages] copies landed + token scales packed
  uint64_t* empty = bars + cfg::kMaxStages;      // [kMaxStages] MMAs done reading the stage
  uint64_t* accf = bars + 2 * cfg::kMaxStages;   // [2] accumulator ready
  uint64_t* acce = accf + 2;                     // [2] accumulator drained by the epilogue
  uint64_t* drain = acce + 2;                    // [1] all MMAs of this CTA complete
  uint64_t* stall = drain + 1;                   // [1] never arrived on (testing aid)
  int32_t* s_end = reinterpret_cast<int32_t*>(smem + cfg::kEndOff);
  int32_t* s_gbase = reinterpret_cast<int32_t*>(smem + cfg::kGbaseOff);
  int32_t* s_wbase = reinterpret_cast<int32_t*>(smem + cfg::kWbaseOff);
  int64_t* s_scan = reinterpret_cast<int64_t*>(smem + cfg::kScanOff);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + cfg::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&misc[0]);
  int* abort_flag = &misc[1];
  uint32_t* s_err = reinterpret_cast<uint32_t*>(&misc[2]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // launched as a programmatic dependent of the kernel before it (the routing step): every
  // input may be that kernel's output, so nothing is read before it has completed
  ptx::griddep_wait();
  // deterministic mode: the combine kernel that follows may launch now (it waits for this grid)
  if constexpr (det) ptx::griddep_launch_dependents();
  const int64_t g0 = threadIdx.x < p.E ? p.group_list[threadIdx.x] : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < cfg::kMaxStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 2);  // producer (with bytes) + packer
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&accf[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&acce[b]), 4);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    ptx::mbar_init(ptx::smem_u32(stall), 1);
    *abort_flag = 0;
    *s_err = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane < 4) ptx::prefetch_tensormap(&tmaps.m[lane]);
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), cfg::kTmemCols);
    ptx::tmem_relinquish();
  }
  __syncthreads();
  int tmax;
  const int n_groups = decode_groups<gemm_threads(fp4)>(p, g0, s_end, s_gbase, s_wbase, s_scan, s_err, tmax);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const Groups groups{s_end, s_gbase, s_wbase, p.E, tmax};
  const int stage_bytes = cfg::stage_bytes(tmax, fp4);
  const int n_stages = cfg::n_stages(tmax, fp4);
  const int off_xsf = cfg::off_xsf(fp4), off_x = cfg::off_x(fp4);
  const Ctl ctl{abort_flag, s_err, p.timeout_ns};
  Sched sched;
  sched.init(n_groups, p.NT, p.KB, det, p.split, det && p.reverse_units, groups);
  const uint32_t smem_base = ptx::smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_stream = ptx::l2_evict_first_policy();  // weights read once
      const uint64_t pol_keep = ptx::l2_evict_last_policy();     // tokens (reused by every column tile), and
                                                                 // weights of experts spanning several groups
      int64_t n_fill = 0;  // stages filled; stage s was filled n_fill / n_stages (+1 if s < n_fill % n_stages) times
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      if (p.test_stall) ok = wait_bar<!det>(ptx::smem_u32(stall), 0, ctl);
      Seg sg;
      int e = -1;
      while (ok && sched.next<det>(sg)) {
        int t0, T;
        groups.info(sg.g, e, t0, T);
        const int m = (T + 15) / 16;  // token rows in 16-row units: boxes of 128/64/32/16 rows
        const int ptile = fp4 ? kPrepTileBytes4 : kPrepTileBytes;
        const uint32_t tx = ptile + m * 16 * 128;
        const uint8_t* wsrc = p.prepared + ((int64_t)e * p.NT + sg.j) * p.KB * (int64_t)ptile;
        // sibling groups of the same expert read the same weight tiles shortly after
        const uint64_t pol_w = (s_gbase[e + 1] - s_gbase[e]) > 1 ? pol_keep : pol_stream;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!wait_bar<!det>(ptx::smem_u32(&empty[stage]), phase ^ 1, ctl)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full[stage]);
          const uint32_t sb = smem_base + stage * stage_bytes;
          ptx::mbar_arrive_expect_tx(fb, tx);
          ptx::bulk_g2s(sb, wsrc + (int64_t)kb * ptile, ptile, fb, pol_w);
          // token rows: one 128-row box, or a 64-row box, then 32-row boxes and a
          // last 16-row box for an odd count (measured fastest on this part)
          int row = 0;
          if (m == 8) {
            ptx::tma_load_2d(sb + off_x, &tmaps.m[3], kb * kTileK, t0, fb, pol_keep);
            row = 128;
          } else if (m > 4) {
            ptx::tma_load_2d(sb + off_x, &tmaps.m[2], kb * kTileK, t0, fb, pol_keep);
            row = 64;
          }
          for (; row < m * 16; row += 32) {
            const int last16 = row + 16 == m * 16;
            ptx::tma_load_2d(sb + off_x + row * 128, &tmaps.m[last16 ? 0 : 1], kb * kTileK, t0 + row, fb,
                             pol_keep);
          }
          ++n_fill;
          if (++stage == n_stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (ok) {  // all fills consumed: wait until the MMA warp has released every stage
        for (int s = 0; s < n_stages; ++s) {
          const int64_t fs = n_fill / n_stages + (s < n_fill % n_stages ? 1 : 0);
          if (fs > 0 && !wait_bar<!det>(ptx::smem_u32(&empty[s]), (uint32_t)((fs - 1) & 1), ctl)) break;
        }
      }
      if (*abort_flag) {  // aborted: let every issued copy land before shared memory is released
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
      // Shared-memory descriptors of stage 0; stage s adds s * (stage_bytes >> 4) to their
      // 14-bit start-address field and an MMA's 32-byte K step adds 2 (shared addresses stay
      // below 2^18, so the field never carries into its neighbours).
      const uint64_t dA0 = ptx::smem_desc(smem_base, 16, 1024, ptx::kSwizzle128B);                // weight tile
      const uint64_t dS0 = ptx::smem_desc(smem_base + cfg::kOffWSF, 0, 128, ptx::kSwizzleNone);  // its scales
      constexpr uint64_t kB = (uint64_t)(cfg::off_x(fp4) >> 4);                          // token rows
      constexpr uint64_t kXs = (uint64_t)((cfg::off_xsf(fp4) - cfg::kOffWSF) >> 4);      // token scales
      constexpr uint64_t kHalf = (uint64_t)(kSfChunk >> 4);                               // second scale half
      const uint32_t dstep = (uint32_t)stage_bytes >> 4;
      const uint32_t sf0 = tmem_base + 2 * tmax;  // per-stage scale columns follow the accumulators
      int stage = 0;
      uint32_t phase = 0, doff = 0, sfoff = 0;
      int acc_i = 0;
      Seg sg;
      bool ok = true;
      int e = -1;
      while (ok && sched.next<det>(sg)) {
        int t0, T;
        groups.info(sg.g, e, t0, T);
        const uint32_t npad = (uint32_t)((T + 15) / 16) * 16;
        const uint32_t idesc = p.idesc | ((npad >> 3) << 17);
        const int buf = acc_i & 1;
        const uint32_t aph = (acc_i >> 1) & 1;
        if (!wait_bar<!det>(ptx::smem_u32(&acce[buf]), aph ^ 1, ctl)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * tmax;
        // packed E2M1 is paced by this loop: four stages per iteration cut its fixed cost per
        // stage (C5 shape 667 -> 627 us per call; unrolled 2: 648, 8: 752 as the loop then no
        // longer stays in the instruction cache); no gain for FP8, which HBM paces
#pragma unroll(fp4 ? 4 : 1)
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!wait_bar<!det>(ptx::smem_u32(&full[stage]), phase, ctl)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t dA = dA0 + doff, dS = dS0 + doff;
          const uint32_t sfa = sf0 + sfoff;
          if constexpr (fp4) {
            // two scale halves per operand (32-blocks 0..3 and 4..7 of the 256-K block); MMA q
            // covers 32-blocks 2q, 2q + 1: half q / 2, bytes 2 (q % 2) and 2 (q % 2) + 1
            const uint32_t sfb = sfa + 8;
            ptx::tc_cp_sf(sfa, dS);
            ptx::tc_cp_sf(sfa + 4, dS + kHalf);
            ptx::tc_cp_sf(sfb, dS + kXs);
            ptx::tc_cp_sf(sfb + 4, dS + kXs + kHalf);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t sid = 2u * (uint32_t)(q & 1);
              const uint32_t col = 4u * (uint32_t)(q >> 1);
              ptx::tc_mma_mxf4(d_tmem, dA + 2 * q, dA + kB + 2 * q, idesc | (sid << 4) | (sid << 29), sfa + col,
                               sfb + col, (kb > sg.kb0 || q > 0) ? 1u : 0u);
            }
          } else {
            const uint32_t sfb = sfa + 4;
            ptx::tc_cp_sf(sfa, dS);
            ptx::tc_cp_sf(sfb, dS + kXs);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              ptx::tc_mma_mxf8(d_tmem, dA + 2 * q, dA + kB + 2 * q, idesc | ((uint32_t)q << 4) | ((uint32_t)q << 29),
                               sfa, sfb, (kb > sg.kb0 || q > 0) ? 1u : 0u);
          }
          ptx::tc_commit(ptx::smem_u32(&empty[stage]));
          doff += dstep;
          sfoff += cfg::sf_cols(fp4);
          if (++stage == n_stages) {
            stage = 0;
            phase ^= 1;
            doff = 0;
            sfoff = 0;
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
  } else if (warp >= 6) {
    // ------------------------------------------------------------ token-scale packers
    // Each packer walks the whole (segment, K block) sequence and loads its own items'
    // scale words three of its items before their stages are filled; it waits about one
    // L2 round trip per item.  Where that paces the ring (eight words per lane for packed
    // E2M1) warp 6 fills the even items and warp 7 the odd
    // ones, running the same code (no instruction-cache cost).  (A 256-thread CTA made the
    // FP8 path slower on small problems, so FP8 keeps one packer.)
    constexpr int npk = fp4 ? 2 : 1;
    const int par = warp - 6;
    if (par < npk) {
      PackIter it;
      it.valid = false;
      it.e = -1;
      uint32_t w0[8], w1[8], w2[8];
      bool v0 = pack_next<det>(it, sched, groups) && (par == 0 || pack_next<det>(it, sched, groups));
      pack_load<fp4>(p, it, w0);
      bool v1 = v0 && pack_next<det>(it, sched, groups) && (npk == 1 || pack_next<det>(it, sched, groups));
      pack_load<fp4>(p, it, w1);
      bool v2 = v1 && pack_next<det>(it, sched, groups) && (npk == 1 || pack_next<det>(it, sched, groups));
      pack_load<fp4>(p, it, w2);
      int stage = par;  // item n fills stage n % n_stages (n_stages >= 6)
      uint32_t phase = 0;
      while (v0) {
        if (!warp_wait_bar<!det>(ptx::smem_u32(&empty[stage]), phase ^ 1, ctl)) break;
        uint8_t* xsf = smem + stage * stage_bytes + off_xsf;
#pragma unroll
        for (int r = 0; r < 4; ++r) *reinterpret_cast<uint32_t*>(xsf + 16 * lane + 4 * r) = w0[r];
        if constexpr (fp4) {
#pragma unroll
          for (int r = 0; r < 4; ++r) *reinterpret_cast<uint32_t*>(xsf + kSfChunk + 16 * lane + 4 * r) = w0[4 + r];
        }
        ptx::fence_proxy_async_smem();  // make the generic-proxy stores visible to tcgen05.cp
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&full[stage]));
        stage += npk;
        if (stage >= n_stages) {
          stage -= n_stages;
          phase ^= 1;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          w0[r] = w1[r];
          w1[r] = w2[r];
        }
        v0 = v1;
        v1 = v2;
        v2 = v2 && pack_next<det>(it, sched, groups) && (npk == 1 || pack_next<det>(it, sched, groups));
        pack_load<fp4>(p, it, w2);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int ep_tid = threadIdx.x - 64;
    // the shared add (atomic mode) runs after the first tile's epilogue, in time the epilogue
    // warps spend waiting anyway; at kernel entry its atomics delayed the first weight loads
    bool shared_pending = !det && p.shared != nullptr && p.shared_rows > 0 && p.N > 0;
    if constexpr (det) {
      if (blockIdx.x == 0) build_row_csr(p, s_end[p.E - 1], ep_tid, s_scan);
    }
    // the tile's token rows and logits, [2][128] (double-buffered by tile parity)
    int32_t* s_trow = reinterpret_cast<int32_t*>(smem + cfg::kTokOff);
    float* s_tlg = reinterpret_cast<float*>(smem + cfg::kTokOff + 2 * 128 * 4);
    int acc_i = 0;
    Seg sg;
    bool bad_row = false;
    int e = -1;
    while (sched.next<det>(sg)) {
      int t0, T;
      groups.info(sg.g, e, t0, T);
      const int buf = acc_i & 1;
      // the tile's out rows and logits, one token per epilogue thread, fetched before the
      // accumulator is ready (fetched per 32-token chunk after it, each chunk waited an L2 round
      // trip: 128-token tiles ended their CTA's work several microseconds late).  Every epilogue
      // warp reaches this barrier on every tile (they walk the same items), and a warp that is
      // one tile ahead writes the other buffer.
      if (ep_tid < T) {
        const int row = load_row32(p.row_index, p.row_i32, (int64_t)t0 + ep_tid, p.batch);
        s_trow[buf * 128 + ep_tid] = row;
        s_tlg[buf * 128 + ep_tid] = p.logit ? p.logit[t0 + ep_tid] : 1.f;
        bad_row |= row < 0;
      }
      ptx::bar_sync(1, 128);
      const uint32_t aph = (acc_i >> 1) & 1;
      if (!warp_wait_bar<!det>(ptx::smem_u32(&accf[buf]), aph, ctl)) break;
      ptx::tc_fence_after();
      const int64_t n = (int64_t)sg.j * kTileN + q * 32 + lane;
      const bool n_ok = n < p.N;
      // the bias term is added once per (token, column): by the segment holding K block 0
      const float bias_n = (p.bias != nullptr && sg.kb0 == 0 && n_ok) ? bf16f(p.bias[(int64_t)e * p.N + n]) : 0.f;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * tmax;
      // one loop per mode, so the atomic mode's hot code holds no store path of the
      // deterministic one (the instruction cache is the scarce resource here); the store path
      // takes 8 tokens per TMEM load, a quarter of the unrolled code of 32 (deterministic C5
      // 1150 -> 1147 us; 16 tokens measured no better)
      if constexpr (det) {  // stored into the per-token buffer
        for (int c0 = 0; c0 < T; c0 += 8) {
          uint32_t v[8];
          ptx::tmem_ld_32x32b_x8(taddr + c0, v);
          ptx::tmem_wait_ld();
          if (c0 + 8 >= T) {  // accumulator fully read: hand it back to the MMA warp
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&acce[buf]));
          }
          const int cnt = T - c0 < 8 ? T - c0 : 8;
          const float* lgs = s_tlg + buf * 128 + c0;  // read as broadcasts
          float* y = p.ybuf + ((int64_t)sg.slot * p.M + t0 + c0) * p.N + n;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (jj < cnt && n_ok) y[(int64_t)jj * p.N] = (__uint_as_float(v[jj]) + bias_n) * lgs[jj];
        }
      } else {  // 16 tokens per TMEM load: half the unrolled scatter code of 32, half the TMEM
                // round trips of 8 (32 -> 8 -> 16 tokens: C1 37.5 -> 37.3 -> 37.1 us,
                // C2 80.6 -> 79.9 -> 79.8, C5 1089.1 -> 1088.4 -> 1086.7)
        float* o = p.out + n;
        for (int c0 = 0; c0 < T; c0 += 16) {
          uint32_t v[16];
          ptx::tmem_ld_32x32b_x16(taddr + c0, v);
          ptx::tmem_wait_ld();
          if (c0 + 16 >= T) {  // accumulator fully read: hand it back to the MMA warp
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&acce[buf]));
          }
          const int cnt = T - c0 < 16 ? T - c0 : 16;
          const int32_t* rows = s_trow + buf * 128 + c0;  // read as broadcasts
          const float* lgs = s_tlg + buf * 128 + c0;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            if (jj < cnt) {
              const int row = rows[jj];
              if (n_ok && row >= 0) ptx::red_add_f32(o + (int64_t)row * p.N, (__uint_as_float(v[jj]) + bias_n) * lgs[jj]);
            }
          }
        }
      }
      ++acc_i;
      if (shared_pending) {
        shared_add_slice(p, ep_tid);
        shared_pending = false;
      }
    }
    if (shared_pending) shared_add_slice(p, ep_tid);  // no tile, or the loop left early
    if (bad_row) atomicOr(s_err, kErrBadRowIndex);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, cfg::kTmemCols);
  }
  if (threadIdx.x == 0) {
    p.hdr[1 + blockIdx.x] = *s_err;
    if (blockIdx.x == 0) p.hdr[0] = gridDim.x;
  }
}

int gemm_smem_bytes() { return cfg::kSmemBytes; }

cudaError_t launch_gemm(const TokenMaps& tmaps, const GemmParams& p, int grid, cudaStream_t s) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaSuccess;
    for (auto k : {gemm_kernel<false, false>, gemm_kernel<false, true>, gemm_kernel<true, false>, gemm_kernel<true, true>})
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // programmatic stream serialization: the launch (and block scheduling) may overlap the tail
  // of the previous kernel in the stream when that kernel allows it; the kernel waits for it
  // before reading any input
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid);
  lc.blockDim = dim3(gemm_threads(p.fp4 != 0));
  lc.dynamicSmemBytes = cfg::kSmemBytes;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  auto kernel = p.fp4 ? (p.deterministic ? gemm_kernel<true, true> : gemm_kernel<true, false>)
                     : (p.deterministic ? gemm_kernel<false, true> : gemm_kernel<false, false>);
  return cudaLaunchKernelEx(&lc, kernel, tmaps, p);
}

}  // namespace gmmfr

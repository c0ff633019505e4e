// Auxiliary kernels of MXFP8 grouped-matmul-finalize-routing:
//   - E2M1 (MXFP4) token expansion to E4M3, and the copy of x1 rows to a 16-byte pitch
//     (K % 16 != 0),
//   - weight preparation (one-time re-layout of x2 and its scales into GEMM tiles),
//   - deterministic combine (row-ordered sum of the per-token results; the row CSR
//     of the routed tokens it walks is built inside the grouped GEMM kernel).
#include "common.cuh"
#include "ptx.cuh"

namespace gmmfr {

// ============================================================================ FP4 expansion
// E2M1 code -> the E4M3 code of the same value (0, 0.5, 1, 1.5, 2, 3, 4, 6; sign in bit 3 -> bit 7).
// Every E2M1 value is exactly an E4M3 value, so the expansion is exact.
__device__ __forceinline__ uint8_t e2m1_to_e4m3(uint32_t c) {
  constexpr uint32_t kLo = 0x3C383000u, kHi = 0x4C484440u;  // codes 0..3 and 4..7, one per byte
  const uint32_t m = c & 7;
  const uint32_t v = ((m < 4 ? kLo : kHi) >> (8 * (m & 3))) & 0xFFu;
  return (uint8_t)(v | ((c & 8) << 4));
}

// Eight E2M1 codes (nibble i = element i) -> eight E4M3 bytes: the magnitude selects a byte
// of the table above with a byte permute, the sign a 0x00 or 0x80 byte.
__device__ __forceinline__ uint4 e2m1x16_to_e4m3(uint32_t a, uint32_t b) {
  constexpr uint32_t kLo = 0x3C383000u, kHi = 0x4C484440u;
  uint32_t o[4];
  const uint32_t w[2] = {a, b};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t mag = w[h] & 0x77777777u;         // selectors 0..7, bit 3 clear
    const uint32_t sgn = (w[h] >> 1) & 0x44444444u;  // selector 4 (the 0x80 byte) where the sign is set
    o[2 * h] = __byte_perm(kLo, kHi, mag) | __byte_perm(0u, 0x80u, sgn);
    o[2 * h + 1] = __byte_perm(kLo, kHi, mag >> 16) | __byte_perm(0u, 0x80u, sgn >> 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// packed [n_bytes] (two codes per byte, even element low) -> fp8 [2 * n_bytes]
// n_vec: leading bytes handled 16 at a time (0 when either pointer is not 16-byte aligned)
__global__ void __launch_bounds__(256) expand_fp4_kernel(const uint8_t* packed, uint8_t* fp8, int64_t n_bytes,
                                                         int64_t n_vec) {
  const int64_t n16 = n_vec / 16;
  const int64_t stride = (int64_t)gridDim.x * 256;
  const uint4* in4 = reinterpret_cast<const uint4*>(packed);
  uint4* out4 = reinterpret_cast<uint4*>(fp8);
  int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {  // four independent loads in flight
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(in4 + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      out4[2 * (i + u * stride)] = e2m1x16_to_e4m3(v[u].x, v[u].y);
      out4[2 * (i + u * stride) + 1] = e2m1x16_to_e4m3(v[u].z, v[u].w);
    }
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldg(in4 + i);
    out4[2 * i] = e2m1x16_to_e4m3(v.x, v.y);
    out4[2 * i + 1] = e2m1x16_to_e4m3(v.z, v.w);
  }
  for (int64_t i = n16 * 16 + (int64_t)blockIdx.x * 256 + threadIdx.x; i < n_bytes; i += (int64_t)gridDim.x * 256) {
    const uint32_t byte = packed[i];
    fp8[2 * i] = e2m1_to_e4m3(byte & 15);
    fp8[2 * i + 1] = e2m1_to_e4m3(byte >> 4);
  }
}

cudaError_t launch_expand_fp4(const uint8_t* packed, uint8_t* fp8, int64_t n_bytes, cudaStream_t s) {
  if (n_bytes == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool vec = ((reinterpret_cast<uintptr_t>(packed) | reinterpret_cast<uintptr_t>(fp8)) & 15) == 0;
  const int64_t n_vec = vec ? n_bytes / 16 * 16 : 0;
  const int64_t work = vec ? n_vec / 16 + (n_bytes - n_vec) : n_bytes;
  const int64_t blocks = (work + 255) / 256;
  expand_fp4_kernel<<<(unsigned)(blocks < sms * 4 ? blocks : sms * 4), 256, 0, s>>>(packed, fp8, n_bytes, n_vec);
  return cudaGetLastError();
}

// x1 rows re-laid at a pitch of Kp = K rounded up to 16 bytes (TMA moves rows whose pitch is a
// multiple of 16 bytes): dst[t, k] = x1[t, k] for k < K and 0 for K <= k < Kp.  With `fp4` the
// source rows hold packed E2M1 codes (K/2 bytes, K even) and are expanded to E4M3 on the way.
// Zero codes past K meet zero weight bytes in the prepared tiles, so they add nothing.
__global__ void __launch_bounds__(256) pad_tokens_kernel(const uint8_t* src, uint8_t* dst, int64_t M, int64_t K,
                                                         int64_t Kp, int32_t fp4) {
  const int64_t n = M * Kp;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    const int64_t t = i / Kp, k = i - t * Kp;
    uint8_t v = 0;
    if (k < K) {
      if (fp4) {
        const uint32_t b = src[t * (K / 2) + k / 2];
        v = e2m1_to_e4m3((k & 1) ? b >> 4 : b & 15);
      } else {
        v = src[t * K + k];
      }
    }
    dst[i] = v;
  }
}

cudaError_t launch_pad_tokens(const uint8_t* x1, uint8_t* dst, int64_t M, int64_t K, int64_t Kp, bool fp4,
                              cudaStream_t s) {
  const int64_t n = M * Kp;
  if (n == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (n + 255) / 256;
  pad_tokens_kernel<<<(unsigned)(blocks < sms * 8 ? blocks : sms * 8), 256, 0, s>>>(x1, dst, M, K, Kp, fp4 ? 1 : 0);
  return cudaGetLastError();
}

// ============================================================================ weight prep
// Prepared tile (e, j, kb): 128 output columns n = j*128 + r by 128 K bytes
// k = kb*128 + c, stored as the shared-memory image of a K-major operand with
// the 128-byte swizzle (16-byte chunk c/16 of row r lands at chunk (c/16)^(r%8)),
// then 512 scale bytes: scale of (row r, 32-block q) at 16*(r%32) + 4*(r/32) + q,
// the 32-row x 16-byte block that tcgen05.cp ... 32x128b.warpx4 spreads over the
// four TMEM lane quadrants.  Columns n >= N and K bytes k >= K are zero; their
// scales (and scales of 32-blocks starting at or past K) are 127 (= 1.0).
__global__ void __launch_bounds__(256) prep_kernel(PrepParams p) {
  const int64_t tiles = p.E * p.NT * p.KB;
  const int64_t Ks = p.Ks;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t kb = tile % p.KB;
    const int64_t j = (tile / p.KB) % p.NT;
    const int64_t e = tile / ((int64_t)p.KB * p.NT);
    uint8_t* dst = p.prepared + tile * kPrepTileBytes;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int id = threadIdx.x + it * 256;
      const int r = id & 127, c = id >> 7;  // warp = 32 consecutive rows of one chunk column
      const int64_t n = j * kTileN + r;
      const int64_t k0 = kb * kTileK + c * 16;
      uint8_t b[16];
      if (p.fp4) {  // packed E2M1: along K (transposed) or along N (not transposed)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint8_t v = 0;
          const int64_t k = k0 + i;
          if (n < p.N && k < p.K) {
            const uint32_t byte = p.transpose_x2 ? p.x2[(e * p.N + n) * (p.K / 2) + k / 2]
                                                 : p.x2[(e * p.K + k) * (p.N / 2) + n / 2];
            const int hi = p.transpose_x2 ? (int)(k & 1) : (int)(n & 1);
            v = e2m1_to_e4m3(hi ? byte >> 4 : byte & 15);
          }
          b[i] = v;
        }
      } else if (p.transpose_x2) {  // x2 [E, N, K]: the 16 bytes are contiguous
        const uint8_t* src = p.x2 + (e * p.N + n) * p.K + k0;
        if (n < p.N && k0 + 16 <= p.K && ((reinterpret_cast<uintptr_t>(src) & 15) == 0)) {
          *reinterpret_cast<uint4*>(b) = *reinterpret_cast<const uint4*>(src);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) b[i] = (n < p.N && k0 + i < p.K) ? src[i] : 0;
        }
      } else {  // x2 [E, K, N]: one byte per K row; a warp reads 32 consecutive n of a row
#pragma unroll
        for (int i = 0; i < 16; ++i)
          b[i] = (n < p.N && k0 + i < p.K) ? p.x2[(e * p.K + k0 + i) * p.N + n] : 0;
      }
      *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = *reinterpret_cast<const uint4*>(b);
    }
    const int64_t sbase = p.scale_per_expert ? e * Ks * p.N * 2 : 0;
    for (int id = threadIdx.x; id < kSfChunk; id += 256) {
      const int r = id & 127, q = id >> 7;
      const int64_t n = j * kTileN + r;
      const int64_t g = kb * 4 + q;  // 32-element block index along K
      uint8_t v = 127;
      if (n < p.N && g * 32 < p.K) {
        const int64_t kp = g >> 1, h = g & 1;
        v = p.transpose_x2 ? p.scale[sbase + (n * Ks + kp) * 2 + h] : p.scale[sbase + (kp * p.N + n) * 2 + h];
      }
      dst[kWTileBytes + 16 * (r & 31) + 4 * (r >> 5) + q] = v;
    }
  }
}

// Packed E2M1 tile (e, j, kb) for kind::mxf4: 128 output columns n = j*128 + r by 256 K
// elements k = kb*256 + 2c + h (byte c of row r, h = 0 low nibble, 1 high), swizzled as
// above, then two 512-byte scale chunks: 32-block kb*8 + 4*h2 + q of row r at
// 512*h2 + 16*(r%32) + 4*(r/32) + q.  Zero codes and 127 scales pad past N and K.
__device__ void prep_tile_fp4(const PrepParams& p, int64_t e, int64_t j, int64_t kb, uint8_t* dst) {
  const int64_t Ks = p.Ks;
  const int64_t Kb = p.K / 2;  // packed bytes of one K row (K is even)
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int id = threadIdx.x + it * 256;
    const int r = id & 127, c = id >> 7;
    const int64_t n = j * kTileN + r;
    const int64_t kk0 = kb * (kTileK4 / 2) + c * 16;  // first packed byte along K
    uint8_t b[16];
    if (p.transpose_x2) {  // x2 [E, N, K/2]: the bytes are already K pairs
      const uint8_t* src = p.x2 + (e * p.N + n) * Kb + kk0;
      if (n < p.N && kk0 + 16 <= Kb && ((reinterpret_cast<uintptr_t>(src) & 15) == 0)) {
        *reinterpret_cast<uint4*>(b) = *reinterpret_cast<const uint4*>(src);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) b[i] = (n < p.N && kk0 + i < Kb) ? src[i] : 0;
      }
    } else {  // x2 [E, K, N/2]: nibble n&1 of rows k = 2kk and 2kk + 1
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint32_t v = 0;
        const int64_t kk = kk0 + i;
        if (n < p.N && kk < Kb) {
          const int sh = (int)(n & 1) * 4;
          const uint32_t lo = (p.x2[(e * p.K + 2 * kk) * (p.N / 2) + n / 2] >> sh) & 15u;
          const uint32_t hi = (p.x2[(e * p.K + 2 * kk + 1) * (p.N / 2) + n / 2] >> sh) & 15u;
          v = lo | (hi << 4);
        }
        b[i] = (uint8_t)v;
      }
    }
    *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = *reinterpret_cast<const uint4*>(b);
  }
  const int64_t sbase = p.scale_per_expert ? e * Ks * p.N * 2 : 0;
  for (int id = threadIdx.x; id < 2 * kSfChunk; id += 256) {
    const int r = id & 127, q = id >> 7;  // q = 0..7: 32-block within the 256-K block
    const int64_t n = j * kTileN + r;
    const int64_t g = kb * 8 + q;
    uint8_t v = 127;
    if (n < p.N && g * 32 < p.K) {
      const int64_t kp = g >> 1, h = g & 1;
      v = p.transpose_x2 ? p.scale[sbase + (n * Ks + kp) * 2 + h] : p.scale[sbase + (kp * p.N + n) * 2 + h];
    }
    dst[kWTileBytes + kSfChunk * (q >> 2) + 16 * (r & 31) + 4 * (r >> 5) + (q & 3)] = v;
  }
}

__global__ void __launch_bounds__(256) prep_fp4_kernel(PrepParams p) {
  const int64_t tiles = p.E * p.NT * p.KB;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t kb = tile % p.KB;
    const int64_t j = (tile / p.KB) % p.NT;
    const int64_t e = tile / ((int64_t)p.KB * p.NT);
    prep_tile_fp4(p, e, j, kb, p.prepared + tile * kPrepTileBytes4);
  }
}

cudaError_t launch_prep(const PrepParams& p, cudaStream_t s) {
  const int64_t tiles = p.E * p.NT * p.KB;
  if (tiles == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t grid = tiles < (int64_t)sms * 8 ? tiles : (int64_t)sms * 8;
  if (p.fp4 && p.fp4_native)
    prep_fp4_kernel<<<(unsigned)grid, 256, 0, s>>>(p);
  else
    prep_kernel<<<(unsigned)grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ============================================================================ deterministic combine
constexpr int kCombineThreads = 256;
constexpr int kCombineCap = 2048;  // row segments up to this length are ordered in shared memory

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Four consecutive floats from column n0 on (one 16-byte load when `vec`, i.e. N % 4 == 0 and
// 16-byte aligned rows); columns past N read 0.
template <bool vec>
__device__ __forceinline__ float4 ld4(const float* row, int64_t n0, int64_t N) {
  if constexpr (vec) return n0 < N ? *reinterpret_cast<const float4*>(row + n0) : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 v;
  v.x = n0 < N ? row[n0] : 0.f;
  v.y = n0 + 1 < N ? row[n0 + 1] : 0.f;
  v.z = n0 + 2 < N ? row[n0 + 2] : 0.f;
  v.w = n0 + 3 < N ? row[n0 + 3] : 0.f;
  return v;
}

__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

// c_t for four columns: Y[0][t] + Y[1][t] + ... over the K splits
template <bool vec>
__device__ __forceinline__ float4 token_sum(const CombineParams& p, int t, int64_t n0) {
  float4 v = ld4<vec>(p.ybuf + (int64_t)t * p.N, n0, p.N);
  for (int s = 1; s < p.split; ++s) add4(v, ld4<vec>(p.ybuf + ((int64_t)s * p.M + t) * p.N, n0, p.N));
  return v;
}

// out[r, n] = ((out[r, n] + c_t1) + c_t2) + ... + w * shared[r - offset, n], the tokens
// t1 < t2 < ... of row r in ascending order, c_t = Y[0][t][n] + Y[1][t][n] + ...
// vec: N % 4 == 0 with 16-byte aligned out and Y rows and 8-byte aligned shared_input rows
template <bool vec>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
  __shared__ int32_t s_tok[kCombineCap];
  __shared__ int32_t s_ord[kCombineCap];
  __shared__ int32_t s_min[kCombineThreads / 32];
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t n0 = ((int64_t)blockIdx.y * kCombineThreads + tid) * 4;
  // out and shared_input are not written by the grouped GEMM in this mode (it writes Y and
  // the row CSR only), so this block reads them while that kernel may still be running
  float4 acc = ld4<vec>(p.out + r * p.N, n0, p.N);
  const bool has_shared = p.shared && r >= p.shared_offset && r < p.shared_offset + p.shared_rows;
  uint2 sh = make_uint2(0, 0);  // four bf16 values, low half first
  if (has_shared) {
    const uint16_t* srow = p.shared + (r - p.shared_offset) * p.N;
    if constexpr (vec) {
      if (n0 < p.N) sh = *reinterpret_cast<const uint2*>(srow + n0);
    } else {
      sh.x = (n0 < p.N ? srow[n0] : 0u) | (n0 + 1 < p.N ? (uint32_t)srow[n0 + 1] << 16 : 0u);
      sh.y = (n0 + 2 < p.N ? srow[n0 + 2] : 0u) | (n0 + 3 < p.N ? (uint32_t)srow[n0 + 3] << 16 : 0u);
    }
  }
  // launched as a programmatic dependent of the grouped GEMM: Y and the row CSR are read only
  // after that kernel has completed
  ptx::griddep_wait();
  const int beg = p.row_ptr[r];
  const int L = p.row_ptr[r + 1] - beg;
  const bool in_smem = L <= kCombineCap;
  if (in_smem) {
    for (int i = tid; i < L; i += kCombineThreads) s_tok[i] = p.sorted[beg + i];
    __syncthreads();
    for (int i = tid; i < L; i += kCombineThreads) {  // rank of a token = number of smaller tokens
      const int t = s_tok[i];
      int rank = 0;
      for (int j = 0; j < L; ++j) rank += s_tok[j] < t;
      s_ord[rank] = t;
    }
    __syncthreads();
    // two tokens' loads in flight at a time; the sums stay in ascending token order
    int i = 0;
    for (; i + 1 < L; i += 2) {
      const float4 a = token_sum<vec>(p, s_ord[i], n0);
      const float4 b = token_sum<vec>(p, s_ord[i + 1], n0);
      add4(acc, a);
      add4(acc, b);
    }
    if (i < L) add4(acc, token_sum<vec>(p, s_ord[i], n0));
  } else {
    int prev = -1;
    for (int i = 0; i < L; ++i) {  // long segment: select the next larger token with a block-wide minimum
      int m = 0x7fffffff;
      for (int j = tid; j < L; j += kCombineThreads) {
        const int u = p.sorted[beg + j];
        if (u > prev && u < m) m = u;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
      if ((tid & 31) == 0) s_min[tid >> 5] = m;
      __syncthreads();
      m = s_min[0];
      for (int w = 1; w < kCombineThreads / 32; ++w) m = min(m, s_min[w]);
      __syncthreads();
      prev = m;
      add4(acc, token_sum<vec>(p, m, n0));
    }
  }
  if (has_shared) {
    acc.x += p.shared_weight * bf16_to_f32(sh.x & 0xFFFF);
    acc.y += p.shared_weight * bf16_to_f32(sh.x >> 16);
    acc.z += p.shared_weight * bf16_to_f32(sh.y & 0xFFFF);
    acc.w += p.shared_weight * bf16_to_f32(sh.y >> 16);
  }
  float* orow = p.out + r * p.N;
  if constexpr (vec) {
    if (n0 < p.N) *reinterpret_cast<float4*>(orow + n0) = acc;
  } else {
    const float a[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (n0 + c < p.N) orow[n0 + c] = a[c];
  }
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  if (p.batch == 0 || p.N == 0) return cudaSuccess;
  const int64_t cols = (p.N + 4 * kCombineThreads - 1) / (4 * kCombineThreads);
  // programmatic stream serialization: the launch overlaps the GEMM's tail (the GEMM lets it
  // start early); the kernel waits for the GEMM before reading anything
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)p.batch, (unsigned)cols);
  lc.blockDim = dim3(kCombineThreads);
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  // 16-byte loads and stores of out and Y rows, 8-byte loads of shared_input rows
  const bool vec = p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(p.out) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(p.ybuf) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(p.shared) & 7) == 0;
  return vec ? cudaLaunchKernelEx(&lc, combine_kernel<true>, p) : cudaLaunchKernelEx(&lc, combine_kernel<false>, p);
}

}  // namespace gmmfr

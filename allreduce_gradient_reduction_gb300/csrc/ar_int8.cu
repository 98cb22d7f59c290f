// 8-bit quantised AllReduce with error feedback.
//
// "Allreduce：大模型分布式训练的核心通信算法与优化实践" §4.2: gradients travel
// as 8-bit integers and are dequantised by the receiver; error feedback adds
// this round's compression error to the next round's gradient.  The pages fix
// nothing further; the block scheme (declared in include/ar.h) is:
//   y = x + e;  per 128-element block  s = max|y| / 127;
//   q = round-half-even(y / s) clamped to [-127, 127] (0 when s = 0);
//   y^ = q * s;  e' = y - y^;
//   the owner of chunk c folds y^ of all ranks in ring order x[c+1], ..., x[c]
//   (AVG: divides by N), requantises the result per block cut at the chunk's
//   ends, and every rank keeps q * s of that.
// Everything is binary32 with explicit round-to-nearest intrinsics, so no
// multiply-add is contracted and the result is bit-identical to the oracle.
//
// One warp owns one 128-element block: 4 consecutive floats per lane (one
// 16-byte access per rank and array), warp shuffles give the block maxima.
#include "ar_fused.cuh"

namespace ar {

constexpr int kQ8 = 128;
constexpr int kQ8Block = 256;  // threads per block: 8 warps, 8 quantisation blocks
constexpr int kQ8Group = 8;    // ranks whose loads are in flight together

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// the 8-bit code, as a float: through an integer, so a code of zero is +0
__device__ __forceinline__ float q8_code(float y, float s) {
  if (s == 0.0f) return 0.0f;
  const int q = __float2int_rn(__fdiv_rn(y, s));  // round half to even; |y / s| <= 127 (+ rounding)
  return (float)min(max(q, -127), 127);
}

__device__ __forceinline__ int chunk_of(int64_t e, int64_t count, int n) {
  return (int)(((e + 1) * n - 1) / count);  // the chunk [floor(cD/N), floor((c+1)D/N)) holding e
}

struct Lane4 {
  float v[4];
};

__device__ __forceinline__ Lane4 load4(const float* p, int64_t e0, int64_t count, bool vec) {
  Lane4 r;
  if (vec && e0 + 3 < count) {
    const float4 t = __ldcg(reinterpret_cast<const float4*>(p + e0));
    r.v[0] = t.x, r.v[1] = t.y, r.v[2] = t.z, r.v[3] = t.w;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) r.v[k] = e0 + k < count ? __ldcg(p + e0 + k) : 0.0f;
  }
  return r;
}

__device__ __forceinline__ void store4(float* p, int64_t e0, int64_t count, bool vec, const Lane4& r) {
  if (vec && e0 + 3 < count) {
    __stcg(reinterpret_cast<float4*>(p + e0), make_float4(r.v[0], r.v[1], r.v[2], r.v[3]));
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (e0 + k < count) __stcg(p + e0 + k, r.v[k]);
  }
}

// y = x + e for one rank, its block scale, the dequantised values; writes e'
__device__ __forceinline__ Lane4 encode(const Lane4& x, const Lane4& e, float* ep, int64_t e0, int64_t count,
                                        bool vec) {
  Lane4 y, yh, en;
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    y.v[k] = __fadd_rn(x.v[k], e.v[k]);
    m = fmaxf(m, fabsf(y.v[k]));
  }
  const float s = __fdiv_rn(warp_max(m), 127.0f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    yh.v[k] = __fmul_rn(q8_code(y.v[k], s), s);
    en.v[k] = __fsub_rn(y.v[k], yh.v[k]);
  }
  store4(ep, e0, count, vec, en);
  return yh;
}

__global__ void __launch_bounds__(kQ8Block, 2) int8_ef_kernel(const __grid_constant__ Int8Args a) {
  __shared__ float s_scale[kQ8Block / 32][kMaxRanks];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t count = a.count;
  const int n = a.nranks;
  const bool vec = a.vec != 0;
  const int64_t nq = (count + kQ8 - 1) / kQ8;
  for (int64_t qb = (int64_t)blockIdx.x * (kQ8Block / 32) + warp; qb < nq;  // this warp's quantisation block
       qb += (int64_t)gridDim.x * (kQ8Block / 32)) {
  const int64_t b0 = qb * kQ8, e0 = b0 + lane * 4;
  const int64_t blast = b0 + kQ8 - 1 < count ? b0 + kQ8 - 1 : count - 1;
  const int c_first = chunk_of(b0, count, n), c_last = chunk_of(blast, count, n);
  float acc[4];

  if (c_first == c_last) {
    // the whole block is in chunk c: fold the ranks in ring order as they come
    const int c = c_first;
    for (int p0 = 0; p0 < n; p0 += kQ8Group) {
      Lane4 xs[kQ8Group], es[kQ8Group];
#pragma unroll
      for (int g = 0; g < kQ8Group; ++g) {  // loads of up to kQ8Group ranks in flight
        if (p0 + g < n) {
          const int r = rot(c + 1 + p0 + g, n);
          xs[g] = load4(a.x[r], e0, count, vec);
          es[g] = load4(a.e[r], e0, count, vec);
        }
      }
#pragma unroll
      for (int g = 0; g < kQ8Group; ++g) {
        if (p0 + g < n) {
          const int r = rot(c + 1 + p0 + g, n);
          const Lane4 yh = encode(xs[g], es[g], a.e[r], e0, count, vec);
#pragma unroll
          for (int k = 0; k < 4; ++k) acc[k] = p0 + g == 0 ? yh.v[k] : __fadd_rn(acc[k], yh.v[k]);
        }
      }
    }
  } else {
    // the block straddles chunks: first every rank's block scale, then each
    // element folds the ranks in the ring order of its own chunk
    for (int r = 0; r < n; ++r) {
      const Lane4 x = load4(a.x[r], e0, count, vec), e = load4(a.e[r], e0, count, vec);
      float m = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) m = fmaxf(m, fabsf(__fadd_rn(x.v[k], e.v[k])));
      m = warp_max(m);
      if (lane == 0) s_scale[warp][r] = __fdiv_rn(m, 127.0f);
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t el = e0 + k;
      if (el >= count) {
        acc[k] = 0.0f;
        continue;
      }
      const int c = chunk_of(el, count, n);
      for (int p = 0; p < n; ++p) {
        const int r = rot(c + 1 + p, n);
        const float y = __fadd_rn(__ldcg(a.x[r] + el), __ldcg(a.e[r] + el));
        const float s = s_scale[warp][r];
        const float yh = __fmul_rn(q8_code(y, s), s);
        __stcg(a.e[r] + el, __fsub_rn(y, yh));
        acc[k] = p == 0 ? yh : __fadd_rn(acc[k], yh);
      }
    }
  }

  if (a.avg) {
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = __fdiv_rn(acc[k], a.fn);
  }
  // requantise: one scale per (block, chunk) piece
  Lane4 res;
  for (int c = c_first; c <= c_last; ++c) {
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (e0 + k < count && (c_first == c_last || chunk_of(e0 + k, count, n) == c)) m = fmaxf(m, fabsf(acc[k]));
    const float s = __fdiv_rn(warp_max(m), 127.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (c_first == c_last || (e0 + k < count && chunk_of(e0 + k, count, n) == c))
        res.v[k] = __fmul_rn(q8_code(acc[k], s), s);
  }
  for (int r = 0; r < n; ++r) store4(a.x[r], e0, count, vec, res);
  __syncwarp();  // s_scale is reused by the warp's next block
  }
}

cudaError_t launch_int8_ef(Int8Args& a, cudaStream_t stream) {
  const int64_t nq = (a.count + kQ8 - 1) / kQ8;
  if (nq == 0) return cudaSuccess;
  const int64_t grid = (nq + kQ8Block / 32 - 1) / (kQ8Block / 32);
  int8_ef_kernel<<<grid_for(grid), kQ8Block, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace ar

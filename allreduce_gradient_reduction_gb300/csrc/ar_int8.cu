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
// Ranks are taken one at a time.  Their loads run ahead of the arithmetic:
// each lane copies its 16 bytes of x and e for the next ranks straight into
// its own shared-memory slots with cp.async, so the copies in flight hold no
// registers and 48 warps per SM still fit (40 registers a thread).
#include "ar_fused.cuh"

namespace ar {

constexpr int kQ8 = 128;
constexpr int kQ8Block = 256;  // threads per block: 8 warps, 8 quantisation blocks
constexpr int kQ8MinBlocks = 6; // resident blocks per SM: 48 warps
constexpr int kQ8Stages = 3;    // ranks whose x and e a warp has in flight or waiting in shared memory

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

// The same code from a reciprocal: t = y * RN(1/s) lies within 1.5 * 2^-23 |y/s|
// of the correctly rounded quotient RN(y/s) (two roundings of 2^-24 each,
// plus RN(y/s)'s own).  When t is farther than |t| * 2^-18 from every
// half-integer, RN(y/s) rounds to the same integer as t, and t is rounded
// with the classic add-and-subtract of 1.5 * 2^23 (exact round-half-even for
// |t| < 2^22; a result of zero comes out +0, as the integer path gives).
// Anything else (near a tie, s = 0 or a non-finite t) takes q8_code itself.
// Saves the per-element divide and the float-int-float round trip.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

__device__ __forceinline__ float q8_code_recip(float y, float s, float r) {
  const float t = __fmul_rn(y, r);
  const float k = __fsub_rn(__fadd_rn(t, kRoundMagic), kRoundMagic);
  const float at = fabsf(t);
  const float slack = __fsub_rn(0.5f, fabsf(__fsub_rn(t, k)));
  if (!(at < 256.0f) || !(slack > __fmul_rn(at, 0x1p-18f))) return q8_code(y, s);
  return fminf(fmaxf(k, -127.0f), 127.0f);
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
  const float rs = __frcp_rn(s);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    yh.v[k] = __fmul_rn(q8_code_recip(y.v[k], s, rs), s);
    en.v[k] = __fsub_rn(y.v[k], yh.v[k]);
  }
  store4(ep, e0, count, vec, en);
  return yh;
}

__global__ void __launch_bounds__(kQ8Block, kQ8MinBlocks) int8_ef_kernel(const __grid_constant__ Int8Args a) {
  __shared__ float s_scale[kQ8Block / 32][kMaxRanks];
  __shared__ float4 s_stage[kQ8Block / 32][kQ8Stages][2][32];  // [warp][slot][x or e][lane]
  pdl_prologue();
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

  if (c_first == c_last && vec && b0 + kQ8 <= count) {
    // a whole aligned block in chunk c: fold the ranks in ring order as they
    // come, the copies of the next kQ8Stages - 1 ranks in flight.  Each lane
    // reads back only the 16 bytes it copied itself, so waiting on its own
    // groups is enough; the slot refilled in step p was read in step p - 1,
    // whose results were stored before this copy is issued.
    const int c = c_first;
    float4 (*st)[2][32] = s_stage[warp];
#pragma unroll
    for (int j = 0; j < kQ8Stages - 1; ++j) {
      if (j < n) {
        const int r = rot(c + 1 + j, n);
        cp_async16(&st[j][0][lane], a.x[r] + e0);
        cp_async16(&st[j][1][lane], a.e[r] + e0);
      }
      cp_async_commit();
    }
    for (int p = 0; p < n; ++p) {
      const int j = p + kQ8Stages - 1;
      if (j < n) {
        const int r = rot(c + 1 + j, n);
        cp_async16(&st[j % kQ8Stages][0][lane], a.x[r] + e0);
        cp_async16(&st[j % kQ8Stages][1][lane], a.e[r] + e0);
      }
      cp_async_commit();  // possibly empty, so that group p is always kQ8Stages - 1 behind
      cp_async_wait<kQ8Stages - 1>();
      const int r = rot(c + 1 + p, n);
      const float4 xv = st[p % kQ8Stages][0][lane], ev = st[p % kQ8Stages][1][lane];
      const Lane4 yh = encode(Lane4{{xv.x, xv.y, xv.z, xv.w}}, Lane4{{ev.x, ev.y, ev.z, ev.w}}, a.e[r], e0, count,
                              true);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = p == 0 ? yh.v[k] : __fadd_rn(acc[k], yh.v[k]);
    }
  } else if (c_first == c_last) {
    // the same from registers: unaligned rows and the ragged last block
    const int c = c_first;
    for (int p = 0; p < n; ++p) {
      const int r = rot(c + 1 + p, n);
      const Lane4 yh = encode(load4(a.x[r], e0, count, vec), load4(a.e[r], e0, count, vec), a.e[r], e0, count, vec);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = p == 0 ? yh.v[k] : __fadd_rn(acc[k], yh.v[k]);
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
    const float rs = __frcp_rn(s);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (c_first == c_last || (e0 + k < count && chunk_of(e0 + k, count, n) == c))
        res.v[k] = __fmul_rn(q8_code_recip(acc[k], s, rs), s);
  }
  for (int r = 0; r < n; ++r) store4(a.x[r], e0, count, vec, res);
  __syncwarp();  // s_scale is reused by the warp's next block
  }
}

cudaError_t launch_int8_ef(Int8Args& a, cudaStream_t stream) {
  const int64_t nq = (a.count + kQ8 - 1) / kQ8;
  if (nq == 0) return cudaSuccess;
  const int64_t grid = (nq + kQ8Block / 32 - 1) / (kQ8Block / 32);
  count_launch();
  return launch_pdl(int8_ef_kernel, grid_for(grid), kQ8Block, stream, a);
}

}  // namespace ar

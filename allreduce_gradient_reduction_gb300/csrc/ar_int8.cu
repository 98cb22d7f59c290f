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
// One warp owns one 128-element block: 4 consecutive floats per lane, warp
// shuffles give the block maxima.  Two kernels share that per-block code:
//  - int8_ef_staged_kernel (16-byte aligned buffers, N <= 8): a persistent
//    block per SM whose producer thread streams super-blocks of 1024
//    elements of every rank's x and e into shared memory with bulk
//    asynchronous copies (cp.async.bulk, completion on an mbarrier), three
//    stages deep, while 8 consumer warps quantise and fold the stage before;
//  - int8_ef_kernel for everything else (and the ragged tail): one rank at a
//    time from global memory, the load latency hidden by 48 resident warps.
#include <atomic>

#include "ar_fused.cuh"

namespace ar {

constexpr int kQ8 = 128;
constexpr int kQ8Block = 256;   // threads per block: 8 warps, 8 quantisation blocks
constexpr int kQ8MinBlocks = 6; // resident blocks per SM: 48 warps hide the loads of a rank at a time

constexpr int kQ8Consumers = 8;                      // consumer warps of the staged kernel
constexpr int kQ8Super = kQ8 * kQ8Consumers;         // elements per rank and array in one stage
constexpr int kQ8StagedThreads = 32 * (kQ8Consumers + 1);
constexpr int kQ8StagedMaxRanks = 8;
constexpr int kQ8SmemBudget = 200 * 1024;            // stages of 2 N kQ8Super floats fit in this
constexpr int kQ8MaxStages = 4;
constexpr unsigned kQ8MaxSpin = 1u << 24;            // backstop if the global timer misbehaves
constexpr int kQ8TimeoutStatus = -4;                 // AR_ERR_TIMEOUT

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

// One warp's quantisation block qb: encode every rank (residuals written
// back), fold in ring order, requantise, store the result to every rank.
// `ld(r, which)` returns this lane's 4 values of rank r's x (which = 0) or
// e (which = 1); `s_scale` is this warp's kMaxRanks floats of shared memory.
template <class Load>
__device__ __forceinline__ void q8_block(const Int8Args& a, int64_t qb, int lane, float* s_scale, Load ld) {
  const int64_t count = a.count;
  const int n = a.nranks;
  const bool vec = a.vec != 0;
  const int64_t b0 = qb * kQ8, e0 = b0 + lane * 4;
  const int64_t blast = b0 + kQ8 - 1 < count ? b0 + kQ8 - 1 : count - 1;
  const int c_first = chunk_of(b0, count, n), c_last = chunk_of(blast, count, n);
  float acc[4];

  if (c_first == c_last) {
    // the whole block is in chunk c: fold the ranks in ring order as they come
    const int c = c_first;
    for (int p = 0; p < n; ++p) {
      const int r = rot(c + 1 + p, n);
      const Lane4 yh = encode(ld(r, 0), ld(r, 1), a.e[r], e0, count, vec);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = p == 0 ? yh.v[k] : __fadd_rn(acc[k], yh.v[k]);
    }
  } else {
    // the block straddles chunks: first every rank's block scale, then each
    // element folds the ranks in the ring order of its own chunk
    for (int r = 0; r < n; ++r) {
      const Lane4 x = ld(r, 0), e = ld(r, 1);
      float m = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (e0 + k < count) m = fmaxf(m, fabsf(__fadd_rn(x.v[k], e.v[k])));
      m = warp_max(m);
      if (lane == 0) s_scale[r] = __fdiv_rn(m, 127.0f);
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
        const float y = __fadd_rn(ld(r, 0).v[k], ld(r, 1).v[k]);  // element el of rank r (its e not yet rewritten)
        const float s = s_scale[r];
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

// ---- register kernel: any alignment, any N, and the staged kernel's tail ----

__global__ void __launch_bounds__(kQ8Block, kQ8MinBlocks) int8_ef_kernel(const __grid_constant__ Int8Args a) {
  __shared__ float s_scale[kQ8Block / 32][kMaxRanks];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nq = (a.count + kQ8 - 1) / kQ8;
  const bool vec = a.vec != 0;
  for (int64_t qb = a.qb_begin + (int64_t)blockIdx.x * (kQ8Block / 32) + warp; qb < nq;
       qb += (int64_t)gridDim.x * (kQ8Block / 32)) {
    const int64_t e0 = qb * kQ8 + lane * 4;
    q8_block(a, qb, lane, s_scale[warp], [&](int r, int which) {
      return load4(which ? a.e[r] : a.x[r], e0, a.count, vec);
    });
  }
}

// ---- staged kernel: bulk asynchronous copies into a 3-deep shared ring -----

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t q8_global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Bounded:
// gives up (false) when `abort` is raised by another warp, after timeout_ns
// of the global timer, or after kQ8MaxSpin polls.
__device__ bool mbar_wait(uint64_t* bar, unsigned parity, const volatile int* abort, int64_t timeout_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = q8_global_ns();
  for (unsigned spins = 0; spins < kQ8MaxSpin; ++spins) {
    if (mbar_test(bar, parity)) return true;
    if ((spins & 63) == 63 && (*abort || q8_global_ns() - t0 > (uint64_t)timeout_ns)) return false;
  }
  return false;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Shared memory: stages x [2N rows of kQ8Super floats] (row 2r = x[r], row
// 2r+1 = e[r] of the stage's super-block), then full[stages] and
// empty[stages] mbarriers, the abort flag and the consumers' scale rows.
struct StagedLayout {
  int stages;
  size_t stage_bytes, bars, bytes;
  __host__ __device__ StagedLayout(int n, int st) : stages(st) {
    stage_bytes = (size_t)2 * n * kQ8Super * sizeof(float);
    bars = stage_bytes * st;
    bytes = bars + 2 * st * sizeof(uint64_t) + 16 + kQ8Consumers * kMaxRanks * sizeof(float);
  }
};

__global__ void __launch_bounds__(kQ8StagedThreads, 1)
    int8_ef_staged_kernel(const __grid_constant__ Int8Args a, int64_t nsuper, int stages) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int n = a.nranks;
  const StagedLayout L(n, stages);
  float* rows = reinterpret_cast<float*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + stages;
  int* abort_flag = reinterpret_cast<int*>(empty + stages);
  float* scales = reinterpret_cast<float*>(smem + L.bars + 2 * stages * sizeof(uint64_t) + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t stage_floats = L.stage_bytes / sizeof(float);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kQ8Consumers);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int* abort_v = abort_flag;

  if (warp == 0) {
    if (lane != 0) return;
    // producer: fill stage it % stages with super-block sb once its consumers released it
    int it = 0;
    bool ok = true;
    for (int64_t sb = blockIdx.x; sb < nsuper; sb += gridDim.x, ++it) {
      const int st = it % stages;
      if (!mbar_wait(&empty[st], ((it / stages) & 1) ^ 1, abort_v, a.timeout_ns)) {
        ok = false;
        break;
      }
      if (blockIdx.x == 0 && it == a.skip_fill) continue;  // test hook: this fill never comes
      mbar_expect_tx(&full[st], (unsigned)L.stage_bytes);
      float* dst = rows + st * stage_floats;
      const int64_t off = sb * kQ8Super;
      for (int r = 0; r < n; ++r) {
        bulk_g2s(dst + (2 * r) * kQ8Super, a.x[r] + off, kQ8Super * sizeof(float), &full[st]);
        bulk_g2s(dst + (2 * r + 1) * kQ8Super, a.e[r] + off, kQ8Super * sizeof(float), &full[st]);
      }
    }
    if (!ok) {
      *abort_v = 1;
      atomicCAS(a.status, 0, kQ8TimeoutStatus);
    }
    // no copy may still be landing in shared memory when the block exits:
    // wait (bounded again) for the last fill of every stage
    const int first = it > stages ? it - stages : 0;
    for (int k = first; k < it; ++k) {
      const volatile int never = 0;
      if (!mbar_wait(&full[k % stages], (k / stages) & 1, &never, a.timeout_ns))
        atomicCAS(a.status, 0, kQ8TimeoutStatus);
    }
    return;
  }

  // consumers: warp c handles quantisation block c of every stage
  const int c = warp - 1;
  float* s_scale = scales + c * kMaxRanks;
  int it = 0;
  for (int64_t sb = blockIdx.x; sb < nsuper; sb += gridDim.x, ++it) {
    const int st = it % stages;
    if (!mbar_wait(&full[st], (it / stages) & 1, abort_v, a.timeout_ns)) {
      if (lane == 0) {
        *abort_v = 1;
        atomicCAS(a.status, 0, kQ8TimeoutStatus);
      }
      return;
    }
    const float* base = rows + st * stage_floats + c * kQ8 + lane * 4;
    q8_block(a, sb * kQ8Consumers + c, lane, s_scale, [&](int r, int which) {
      const float4 t = *reinterpret_cast<const float4*>(base + (2 * r + which) * kQ8Super);
      Lane4 v;
      v.v[0] = t.x, v.v[1] = t.y, v.v[2] = t.z, v.v[3] = t.w;
      return v;
    });
    if (lane == 0) mbar_arrive(&empty[st]);  // q8_block ended with __syncwarp: the warp is done with the stage
  }
}

static int staged_stages(int n) {
  const StagedLayout one(n, 1);
  int st = (int)(kQ8SmemBudget / one.stage_bytes);
  return st > kQ8MaxStages ? kQ8MaxStages : st;
}

// Opens the staged kernel up to the largest shared memory any N <= 8 needs,
// once per device.
static cudaError_t open_staged_smem() {
  static std::atomic<bool> opened[256];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
  if (opened[dev].load()) return cudaSuccess;
  size_t most = 0;
  for (int n = 1; n <= kQ8StagedMaxRanks; ++n) {
    const StagedLayout L(n, staged_stages(n));
    if (L.bytes > most) most = L.bytes;
  }
  e = cudaFuncSetAttribute(int8_ef_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
  if (e == cudaSuccess) opened[dev].store(true);
  return e;
}

cudaError_t launch_int8_ef(Int8Args& a, cudaStream_t stream) {
  const int64_t nq = (a.count + kQ8 - 1) / kQ8;
  if (nq == 0) return cudaSuccess;
  a.qb_begin = 0;
  const int64_t nsuper = a.vec && a.nranks <= kQ8StagedMaxRanks ? a.count / kQ8Super : 0;
  const int stages = staged_stages(a.nranks);
  if (nsuper > 0 && stages >= 2) {
    const StagedLayout L(a.nranks, stages);
    cudaError_t e = open_staged_smem();
    if (e != cudaSuccess) return e;
    const int64_t grid = nsuper < sm_count() ? nsuper : sm_count();
    int8_ef_staged_kernel<<<(unsigned)grid, kQ8StagedThreads, L.bytes, stream>>>(a, nsuper, stages);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    a.qb_begin = nsuper * kQ8Consumers;
    if (a.qb_begin >= nq) return cudaSuccess;
  }
  const int64_t grid = (nq - a.qb_begin + kQ8Block / 32 - 1) / (kQ8Block / 32);
  int8_ef_kernel<<<grid_for(grid), kQ8Block, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace ar

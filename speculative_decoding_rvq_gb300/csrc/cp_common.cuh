// cp_common.cuh -- device helpers shared by the kernels of the CUDA library.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cpk {

// ---------------------------------------------------------------- Philox
// Philox4x32-10 written from its published definition (Salmon, Moraes,
// Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11):
// round (x0..x3) -> (hi(M1*x2) ^ x1 ^ k0, lo(M1*x2), hi(M0*x0) ^ x3 ^ k1,
// lo(M0*x0)), key bumped by the Weyl constants between rounds.
struct Philox {
  static constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  static constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
  __device__ __forceinline__ static uint4 block(uint4 x, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
      if (r) { k.x += kW0; k.y += kW1; }
      const uint32_t lo0 = kM0 * x.x, hi0 = __umulhi(kM0, x.x);
      const uint32_t lo1 = kM1 * x.z, hi1 = __umulhi(kM1, x.z);
      x = make_uint4(hi1 ^ x.y ^ k.x, lo1, hi0 ^ x.w ^ k.y, lo0);
    }
    return x;
  }
};

enum : uint32_t { kDraft = 0, kAccept = 1, kTarget = 2, kTreeAccept = 4 /* + child index */ };

// u in [0, 1): top 24 bits of word 0, exact in float32.
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t stream, uint32_t frame,
                                                uint32_t depth, uint32_t purpose) {
  const uint4 o = Philox::block(make_uint4(stream, frame, depth, purpose),
                                make_uint2((uint32_t)(seed & 0xFFFFFFFFull), (uint32_t)(seed >> 32)));
  return __uint2float_rn(o.x >> 8) * 5.9604644775390625e-08f;  // 2^-24
}

// ----------------------------------------------------------------- memory
// Bulk prefetch of a byte range into L2 (Hopper/Blackwell bulk-copy unit).
// addr and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 16-byte asynchronous global -> shared copy through L2 only (cp.async.cg):
// the data may have been written by other CTAs of the same launch.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Warp-cooperative async copy of `bytes` (multiple of 16, both ends 16-byte
// aligned) from global to shared memory.  Call cp_async_wait_all() and
// __syncwarp() before reading the destination.
__device__ __forceinline__ void warp_copy_async(void* smem_dst, const void* gsrc, int bytes) {
  const int lane = threadIdx.x & 31;
  char* d = static_cast<char*>(smem_dst);
  const char* s = static_cast<const char*>(gsrc);
  for (int o = lane * 16; o < bytes; o += 512) cp_async16(d + o, s + o);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------ mbarrier + bulk copies
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// One arrival that also announces `bytes` of transactions to come.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// An L2 policy under which the lines a copy brings in are the first to be
// evicted.  Weights are read once per pass and the pass streams more bytes
// than L2 holds, so they must not push out what is reused within a pass
// (exchange buffers, KV cache, code).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared by the TMA unit under L2 policy `policy`;
// completion is signalled on `bar` as transaction bytes.  dst, src and bytes
// must be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
               : "memory");
}

// 1-D bulk copy global -> shared without a cache hint (data that other CTAs
// reuse, e.g. activation rows written by the previous kernel).
__device__ __forceinline__ void bulk_copy_g2s_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, bounded by timeout_ns of
// %globaltimer; returns false (after raising the status word) on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) { atomicCAS(status, 0, -5); return false; }
  }
  return true;
}

// Plain arrival (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Inverse of float_key.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}


// bf16x2 word -> two floats (low half = element 0).
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Order-preserving map float -> uint32 (larger float, larger key; -0 < +0).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Device status word values (mirror cp_spec_status).
enum : int { kStatusOk = 0, kStatusTimeout = -5, kStatusDevice = -7 };

__device__ __forceinline__ void raise_status(int* status, int code) { atomicCAS(status, 0, code); }

// ------------------------------------------------------------ arithmetic
// e^d for d <= 0 in float32, the softmax exponential of the sampling path,
// written from the mathematics: Cody-Waite range reduction (Cody and Waite,
// "Software Manual for the Elementary Functions", 1980), n = rint(d log2 e),
// r = d - n ln 2 with ln 2 split into an exact-product high part and a low
// part, the degree-7 Taylor polynomial of e^r by Horner with fused
// multiply-adds, and an exact scaling by 2^n; defined as 0 below d = -87.
// Each step is one IEEE float32 operation (no contraction, no flush to zero),
// so the CPU restatement of the same sequence gives the same bits.
__device__ __forceinline__ float cp_expf(float d) {
  if (!(d >= -87.0f)) return 0.0f;
  const float n = rintf(__fmul_rn(d, 0x1.715476p+0f));
  float r = fmaf(-n, 0x1.62e4p-1f, d);
  r = fmaf(-n, 0x1.7f7d1cp-20f, r);
  float p = 0x1.a01a02p-13f;
  p = fmaf(p, r, 0x1.6c16c2p-10f);
  p = fmaf(p, r, 0x1.111112p-7f);
  p = fmaf(p, r, 0x1.555556p-5f);
  p = fmaf(p, r, 0x1.555556p-3f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  return __fmul_rn(p, __uint_as_float((uint32_t)((int)n + 127) << 23));
}

// Two independent float32 fused multiply-adds in one instruction:
// (c.x + a.x * b.x, c.y + a.y * b.y), each rounded once.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%0, %1};\n"
      " fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0, %1}, rc;\n}"
      : "+f"(c.x), "+f"(c.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return c;
}

}  // namespace cpk

// cp_t5.cuh -- the GEMVs of the pass as fifth-generation tensor-core
// (tcgen05) tiles, for contexts with many rows per pass (many streams).
// Included by cp_pass_kernels.cu inside namespace cpk, after the pass helpers
// it uses.
//
// A GEMV is Y[pass row][unit] = sum_k W[unit row][k] x'[pass row][k] with x'
// the input row (times the RMSNorm gain for the normed kinds; the row's
// RMSNorm scale multiplies the sum).  A CTA computes one tile: kT5M = 128
// weight rows (blockIdx.y) against RB pass rows (blockIdx.x, RB = 16, 32 or
// 64 per kind).  The weight rows are the A operand (M = 128); the pass rows,
// each split into bf16 hi = rn(x') and lo = rn(x' - hi), the B operand: B row
// 2i is the hi part of the tile's pass row i, B row 2i + 1 its lo part, so
// N = 2 RB.  The MMAs (kind::f16, bf16 x bf16 -> fp32) accumulate into N
// TMEM columns; the epilogue reads TMEM lane m (weight row m) and finishes
// y = D[m][2i] + D[m][2i + 1].  For pair kinds (QKV: RoPE pair e, e + d/2 of
// a head; gate/up) A rows 0..63 hold the first rows of the tile's 64 units and
// A rows 64..127 their second rows; the epilogue joins a pair through shared
// memory.
//
// K runs in slabs of 64 elements.  A ring of `stages` stages holds per slab
// the 128 weight rows in the 128-byte-swizzled K-major layout (atoms of 8
// rows x 128 bytes, 16-byte chunk j of row r at chunk j ^ (r mod 8)) and the
// tile's raw input rows (fp32, or bf16 for layer 0's code embeddings).  The
// CTA's warps take three roles, linked by mbarriers:
//   - four copy warps fill a slab's ring stage once the MMAs of the stage's
//     previous slab completed (`empty`): one thread issues the weight boxes
//     as TMA tensor copies (cp.async.bulk.tensor with a 128-byte-swizzled
//     map per weight matrix, 1-4 boxes per slab) with their byte count on
//     the stage's `wfull` barrier, and every copy thread issues cp.async
//     copies of the input rows and arrives on `full` when they landed
//     (cp.async.mbarrier.arrive.noinc), so a slab is released as soon as its
//     data is there, whatever the MMAs are doing;
//   - eight conversion warps turn the raw rows of a slab into one of three B
//     stages (gain, split hi / lo, sums of squares) once the MMAs that read
//     the B stage before completed, and release it (`bfull`);
//   - one warp waits for each converted slab and one of its lanes issues the
//     slab's four k16 MMAs and commits them to the
//     ring stage's `empty` barrier, which both the copy warps (ring stage
//     free) and the conversion warps (B stage free) wait on.
// The conversion warps execute a generic-to-async proxy fence after writing
// a B stage, before handing it on, so their st.shared writes are visible to
// the tensor core (the weight boxes arrive through the async proxy itself).
// Every wait is bounded; a wait that runs out raises the device status and
// an abort flag that ends every other wait of the CTA, and an aborted CTA
// waits (bounded) for its weight boxes still in flight before it exits.  A row's sum of
// squares is 16 partial sums, one per 16-byte chunk column of the slab rows
// (over the slabs in order), added in column order: no reduction order
// depends on the tile height or on which rows share the pass.
//
// The lm_heads tile of head slot j takes only the pass rows that read head
// j (their logit slots), compacted in pass-row order.
#pragma once

constexpr int kT5MaxStages = 6;
constexpr int kT5SlabBytes = kT5M * 128;  // one slab of the weight tile
constexpr int kT5BStages = 3;
constexpr int kT5ConvThreads = 256;       // warps 0-7: conversion and epilogue
constexpr int kT5CopyThreads = 128;       // warps 8-11: copies
constexpr int kT5Threads = kT5ConvThreads + kT5CopyThreads + 32;  // warp 12: MMA issue
constexpr int kT5XRows = 64 * 16 / kT5CopyThreads;   // input rows per copy thread, at most

struct T5Shared {
  uint64_t full[kT5MaxStages];   // ring stage holds its slab's input rows (one arrival per copy thread)
  uint64_t wfull[kT5MaxStages];  // ring stage holds its slab's weight boxes (one arrival plus their bytes)
  uint64_t empty[kT5MaxStages];  // MMAs of the ring stage's slab completed
  uint64_t bfull[kT5BStages];    // B stage converted (one arrival per conversion warp)
  uint64_t dbar;                 // every MMA of the tile completed
  uint64_t hbar;                 // test hook: a barrier nothing arrives on
  int abort;                     // a bounded wait ran out: every role stops
  int nrows, nheads, cnt;
  uint32_t tmem;                 // TMEM accumulator address
  int plan_w[2];
  int heads[kMaxHeadsPerPass];
  CallArgs ca;
};

__device__ __forceinline__ uint64_t t5_sdesc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu)  // start address / 16
         | ((uint64_t)1 << 16)             // leading byte offset (unused for swizzled K-major)
         | ((uint64_t)(1024 >> 4) << 32)   // stride byte offset: 8-row atoms 1024 bytes apart
         | ((uint64_t)1 << 46)             // descriptor version
         | ((uint64_t)2 << 61);            // 128-byte swizzle
}

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both
// K-major, N columns, M = kT5M.
__device__ __forceinline__ uint32_t t5_idesc(int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kT5M >> 4) << 24);
}

// Byte offset of 16-byte chunk j (of 8 per slab row) of row r in a swizzled
// slab.
__device__ __forceinline__ uint32_t t5_swz(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

// bf16x2 hi = rn(x) and lo = rn(x - hi) of a pair.
__device__ __forceinline__ void t5_split(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 o = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&o);
}

// Bounded wait for phase `parity` of `bar` that also ends when another
// thread of the CTA raised the abort flag.  A wait that runs out raises the
// device status (timeout) and the flag.
__device__ __forceinline__ bool t5_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                                        uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort = 1;
      atomicCAS(status, 0, -5);
      return false;
    }
  }
  return true;
}

// Shared-memory carve-up (the host sizes the launch with the same arithmetic).
struct T5Smem {
  size_t a, b, raw, gain, ss, rows, list, wrow, xrow, ep, xch, rope, total;
};
__host__ __device__ inline T5Smem t5_smem_layout(int kind, int RB, int stages, int K, int rows_cap, int G, int d) {
  T5Smem o;
  size_t off = 0;
  o.a = off; off += (size_t)stages * kT5SlabBytes;           // weight slabs (1024-aligned)
  o.b = off; off += (size_t)kT5BStages * RB * 256;           // B stages of 2 RB rows x 128 bytes
  o.raw = off; off += (size_t)stages * RB * 256;             // raw input slabs: RB rows x 64 fp32
  o.gain = off; off += (kind == kQKV || kind == kGU || kind == kHeads) ? (size_t)K * 4 : 0;
  o.ss = off; off += (size_t)(64 * 16 + 64) * 4;            // sums of squares per (row, chunk column), then RMSNorm scales
  o.rows = off; off += (size_t)((3 * rows_cap + 3) / 4 * 4) * 4;
  o.list = off; off += 64 * 4;                               // the tile's pass rows (compacted indices)
  o.wrow = off; off += (size_t)kT5M * 8;                     // global address of each weight row
  o.xrow = off; off += 64 * 8 + 64 * 4;                      // global address and bytes per slab of each input row
  o.ep = off; off += 64 * 24;                                // epilogue: two offsets and the position per row
  o.xch = off; off += 2 * 64 * 8 * 4;                        // epilogue: second rows of the pairs, per warp group
  o.rope = off; off += kind == kQKV && (size_t)G * (d / 2) * 8 <= (size_t)kRopeSmemBytes ? (size_t)kRopeSmemBytes : 0;
  o.total = off + 1024;  // room to align the base to 1024 bytes
  return o;
}

// Weight-row tiles (blockIdx.y) of a GEMV kind with `units` output units.
__host__ __device__ inline int t5_mtiles(int kind, int units) {
  const int rpu = (kind == kQKV || kind == kGU) ? 2 : 1;
  return (units * rpu + kT5M - 1) / kT5M;
}

template <int KIND>
__global__ void __launch_bounds__(kT5Threads, 1) t5_kernel(const __grid_constant__ FrameParams P, int l) {
  extern __shared__ __align__(1024) unsigned char t5smem_raw[];
  pdl_launch_dependents();
  __shared__ T5Shared sh;
  constexpr bool kPair = KIND == kQKV || KIND == kGU;
  constexpr bool kNormed = KIND == kQKV || KIND == kGU || KIND == kHeads;
  constexpr int kRpu = kPair ? 2 : 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = gemv_K(P, KIND), slabs = K / 64;
  const int RB = P.t5_rb[KIND], NST = P.t5_stages[KIND];
  const int N = 2 * RB;
  const int rows_cap = P.Bmax * P.NS;
  const int mt = blockIdx.y, rb = blockIdx.x;
  unsigned char* smem = t5smem_raw + ((1024u - (smem_u32(t5smem_raw) & 1023u)) & 1023u);
  const T5Smem L = t5_smem_layout(KIND, RB, NST, K, rows_cap, P.G, P.d);
  unsigned char* abase = smem + L.a;
  unsigned char* bbase = smem + L.b;
  unsigned char* rawb = smem + L.raw;
  float* s_gain = reinterpret_cast<float*>(smem + L.gain);
  float* s_ss = reinterpret_cast<float*>(smem + L.ss);
  float* s_inv = s_ss + 64 * 16;
  int* s_rows = reinterpret_cast<int*>(smem + L.rows);
  int* s_list = reinterpret_cast<int*>(smem + L.list);
  const unsigned char** s_wrow = reinterpret_cast<const unsigned char**>(smem + L.wrow);
  const unsigned char** s_xrow = reinterpret_cast<const unsigned char**>(smem + L.xrow);
  int* s_xstep = reinterpret_cast<int*>(smem + L.xrow + 64 * 8);
  long long* s_ep = reinterpret_cast<long long*>(smem + L.ep);  // [64][3]: offsets, position
  float2* s_rope = reinterpret_cast<float2*>(smem + L.rope);
  PassRows pr{s_rows, s_rows + rows_cap, s_rows + 2 * rows_cap};
  const size_t rope_n = (size_t)P.G * (P.d / 2);
  const bool rope_in_smem = KIND == kQKV && rope_n * sizeof(float2) <= (size_t)kRopeSmemBytes;
  const float* gain_g = KIND == kQKV ? P.attn_norm[l] : (KIND == kGU ? P.ffn_norm[l] : (KIND == kHeads ? P.final_norm : nullptr));
  const bool need_heads = KIND == kHeads || (KIND == kGU && l == P.L - 1);
  volatile int* abort = &sh.abort;
  // test hook: the MMA thread of CTA (0, 0) of the pass's first GEMV waits on a barrier nothing arrives on
  const bool stall = P.test_stall && KIND == kQKV && l == 0 && mt == 0 && rb == 0;

  // ---------------- before the dependency wait: what no kernel of the pass writes
  if (tid < 2) sh.plan_w[tid] = __ldcg(tid == 0 ? &P.plan->nrows : &P.plan->nheads);
  if (tid == 2) sh.abort = 0;
  if (need_heads && tid >= 32 && tid < 32 + kMaxHeadsPerPass) sh.heads[tid - 32] = __ldcg(&P.plan->heads[tid - 32]);
  if (tid >= 128 && tid < 128 + (int)(sizeof(CallArgs) / 4))
    reinterpret_cast<int*>(&sh.ca)[tid - 128] = __ldcg(reinterpret_cast<const int*>(P.call) + (tid - 128));
  for (int i = tid; i < 3 * rows_cap; i += kT5Threads) {
    const int a = i / rows_cap, j = i - a * rows_cap;
    s_rows[i] = __ldcg((a == 0 ? P.prow : (a == 1 ? P.ppos : P.pcode)) + j);
  }
  __syncthreads();
  const int nrows = min(sh.plan_w[0], rows_cap);
  const int nheads = need_heads ? min(sh.plan_w[1], kMaxHeadsPerPass) : 0;
  const int units = gemv_units(P, KIND, nheads);
  const int u0 = mt * (kT5M / kRpu);                       // first unit of the tile
  const int nun = min(kT5M / kRpu, units - u0);            // units of the tile
  // the tile's pass rows: a block of the pass's rows, or (lm_heads) a block of
  // the rows that read the tile's head
  int cnt;
  if (KIND == kHeads) {
    if (warp == 0 && nun > 0) {
      const int head = sh.heads[u0 / P.V];
      int c = 0;
      for (int b = 0; b < nrows; b += 32) {
        const int i = b + lane;
        const int slot = i < nrows ? head - pr.ppos[i] : -1;
        const bool take = i < nrows && pr.ppos[i] >= 1 && slot >= 0 && slot <= P.ND;
        const unsigned m = __ballot_sync(0xffffffffu, take);
        const int at = c + __popc(m & ((1u << lane) - 1u)) - rb * RB;
        if (take && at >= 0 && at < RB) s_list[at] = i;
        c += __popc(m);
      }
      if (lane == 0) sh.cnt = c;
    }
    __syncthreads();
    cnt = nun > 0 ? min(RB, sh.cnt - rb * RB) : 0;
  } else {
    cnt = nun > 0 ? min(RB, nrows - rb * RB) : 0;
    if (tid < RB) s_list[tid] = rb * RB + tid;
  }
  if (cnt <= 0) return;  // nothing of this tile in the pass (no copy issued, no TMEM held)

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&sh.full[i], kT5CopyThreads);
      mbar_init(&sh.wfull[i], 1);
      mbar_init(&sh.empty[i], 1);
    }
    for (int i = 0; i < kT5BStages; ++i) mbar_init(&sh.bfull[i], kT5ConvThreads / 32);
    mbar_init(&sh.dbar, 1);
    mbar_init(&sh.hbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {  // TMEM accumulator: N columns (a power of two >= 32)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem)),
                 "r"(N) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid < kT5M) {  // global address of A row tid of the tile (null past the tile's rows), for the L2 prefetch
    const int j = u0 + (kPair ? (tid & 63) : tid);
    const bool in = kPair ? (tid & 63) < nun : tid < nun;
    s_wrow[tid] = in ? mv_row_src(P, KIND, l, sh.heads, j, kPair ? (tid >> 6) : 0) : nullptr;
  }
  // RoPE table and norm gain (conversion threads, waited for before the epilogue / conversion)
  if (tid < kT5ConvThreads) {
    if (rope_in_smem)
      for (int i = tid; i < (int)(rope_n / 2); i += kT5ConvThreads) cp_async16(s_rope + 2 * i, P.rope + 2 * i);
    if (gain_g != nullptr)
      for (int i = tid; i < K / 4; i += kT5ConvThreads) cp_async16(s_gain + 4 * i, gain_g + 4 * i);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  __syncthreads();  // barriers initialised, TMEM address, weight rows
  const uint32_t tmem = sh.tmem;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  if (warp >= kT5ConvThreads / 32 && warp < (kT5ConvThreads + kT5CopyThreads) / 32) {
    // ================= copy warps
    const int ct = tid - kT5ConvThreads;
    for (int r = ct; r < nun * kRpu; r += kT5CopyThreads) prefetch_l2(s_wrow[r], (uint32_t)K * 2u);
    // the slab's weight boxes (copy thread 0): map, first row, A row, rows
    int bmap[4], by[4], barow[4], brows[4], nbox = 0;
    if (ct == 0) {
      if (KIND == kQKV) {
        const int half = P.d / 2, nh = 64 / half;
        for (int i = 0; i < nh; ++i) {
          const int hh = u0 / half + i;
          int which, lh;
          if (hh < P.nq) { which = kMapQ; lh = hh; }
          else if (hh < P.nq + P.nkv) { which = kMapK; lh = hh - P.nq; }
          else if (hh < P.nq + 2 * P.nkv) { which = kMapV; lh = hh - P.nq - P.nkv; }
          else break;
          const int map = t5_map_index(P.L, l, which);
          bmap[nbox] = map; by[nbox] = lh * P.d; barow[nbox] = i * half; brows[nbox] = half; ++nbox;
          bmap[nbox] = map; by[nbox] = lh * P.d + half; barow[nbox] = 64 + i * half; brows[nbox] = half; ++nbox;
        }
      } else if (KIND == kGU) {
        bmap[0] = t5_map_index(P.L, l, kMapGate); by[0] = u0; barow[0] = 0; brows[0] = 64;
        bmap[1] = t5_map_index(P.L, l, kMapUp); by[1] = u0; barow[1] = 64; brows[1] = 64;
        nbox = 2;
      } else if (KIND == kHeads) {
        const int hi = u0 / P.V;
        bmap[0] = t5_map_index(P.L, 0, -1); by[0] = (sh.heads[hi] - 1) * P.V + (u0 - hi * P.V); barow[0] = 0;
        brows[0] = kT5M;
        nbox = 1;
      } else {
        bmap[0] = t5_map_index(P.L, l, KIND == kO ? kMapO : kMapDown); by[0] = u0; barow[0] = 0; brows[0] = kT5M;
        nbox = 1;
      }
    }
    uint32_t wbytes = 0;
    for (int q = 0; q < nbox; ++q) {
      wbytes += (uint32_t)brows[q] * 128u;
      // the maps were written to global memory by the host: acquire them for the tensor-map proxy
      asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(P.tmaps + (size_t)bmap[q] * 128)
                   : "memory");
    }
    int last_w = -1;  // the last slab whose weight boxes thread 0 issued
    pdl_wait();
    if (ct < cnt) {  // input row ct of the tile
      const ActRow a = act_row<__nv_bfloat16>(P, sh.ca, pr, KIND, l, s_list[ct]);
      s_xrow[ct] = a.f != nullptr ? reinterpret_cast<const unsigned char*>(a.f) : static_cast<const unsigned char*>(a.w);
      s_xstep[ct] = a.f != nullptr ? 256 : 128;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kT5CopyThreads) : "memory");  // the copy warps' row table
    // input chunks: rows (ct >> 4) + (kT5CopyThreads / 16) q, 16-byte chunk ct & 15 (fp32
    // rows: 16 chunks per slab row; bf16 code embeddings: 8)
    const unsigned char* xsrc[kT5XRows];
    int xsteps[kT5XRows];
#pragma unroll
    for (int q = 0; q < kT5XRows; ++q) {
      const int i = (ct >> 4) + (kT5CopyThreads / 16) * q;
      const bool v = i < cnt && (ct & 15) * 16 < s_xstep[i];
      xsrc[q] = v ? s_xrow[i] + (ct & 15) * 16 : nullptr;
      xsteps[q] = v ? s_xstep[i] : 0;
    }
    const uint32_t xdst = (uint32_t)((ct >> 4) * 256 + (ct & 15) * 16);
    bool ok = true;
    for (int j = 0; j < slabs; ++j) {
      {
        const int st = j % NST;
        if (j >= NST && !t5_wait(&sh.empty[st], (uint32_t)((j / NST) - 1) & 1u, abort, &P.ctl->status, P.wait_ns)) {
          ok = false;
          break;
        }
        if (ct == 0) {  // the weight boxes, their bytes announced on the stage's barrier first
          unsigned char* wst = abase + (size_t)st * kT5SlabBytes;
          const uint32_t bar = smem_u32(&sh.wfull[st]);
          last_w = j;
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(wbytes) : "memory");
          for (int q = 0; q < nbox; ++q)
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                ::"r"(smem_u32(wst + barow[q] * 128)), "l"(P.tmaps + (size_t)bmap[q] * 128), "r"(j * 64), "r"(by[q]),
                  "r"(bar)
                : "memory");
        }
        unsigned char* xst = rawb + (size_t)st * RB * 256 + xdst;
#pragma unroll
        for (int q = 0; q < kT5XRows; ++q)
          if (xsrc[q] != nullptr) cp_async16(xst + q * (kT5CopyThreads * 16), xsrc[q] + (size_t)j * xsteps[q]);
        // one arrival on the stage's barrier once this thread's copies landed
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&sh.full[st])) : "memory");
      }
    }
    cp_async_wait_all();
    if (!ok) {
      // an aborted CTA leaves slabs nobody waits for: the weight boxes of the
      // last slab of each stage complete on their own barrier (bounded wait),
      // and the input copies' arrivals are given time to land
      if (ct == 0)
        for (int j = max(0, last_w - NST + 1); j <= last_w; ++j)
          mbar_wait_bounded(&sh.wfull[j % NST], (uint32_t)(j / NST) & 1u, &P.ctl->status, P.wait_ns);
      __nanosleep(4000);
    }
  } else if (warp == (kT5ConvThreads + kT5CopyThreads) / 32) {
    // ================= MMA warp: the whole warp waits (converged); lane 0 issues
    bool ok = !stall || t5_wait(&sh.hbar, 0, abort, &P.ctl->status, P.wait_ns);
    ok = __all_sync(0xffffffffu, ok);
    const uint32_t idesc = t5_idesc(N);
    for (int s = 0; s < slabs && ok; ++s) {
      const int bs = s % kT5BStages;
      ok = __all_sync(0xffffffffu, t5_wait(&sh.bfull[bs], (uint32_t)(s / kT5BStages) & 1u, abort, &P.ctl->status, P.wait_ns));
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (lane == 0) {
        const uint32_t a0 = smem_u32(abase + (size_t)(s % NST) * kT5SlabBytes);
        const uint32_t b0 = smem_u32(bbase + (size_t)bs * RB * 256);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint64_t ad = t5_sdesc(a0 + c * 32), bd = t5_sdesc(b0 + c * 32);
          const uint32_t acc = (s | c) ? 1u : 0u;
          asm volatile("{\n .reg .pred pa;\n setp.ne.b32 pa, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pa;\n}"
                       ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(acc) : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&sh.empty[s % NST]))
                     : "memory");
      }
      __syncwarp();
    }
    // every MMA issued (or none) completes before the barrier's phase does
    if (lane == 0)
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&sh.dbar))
                   : "memory");
    __syncwarp();
    if (!ok && lane == 0) mbar_wait_bounded(&sh.dbar, 0, &P.ctl->status, P.wait_ns);  // nothing in flight at exit
  } else {
    // ================= conversion warps (then the epilogue)
    pdl_wait();
    if (KIND == kQKV && l == 0) {
      // the residual stream starts as the input rows: this CTA's rows, its slice of H
      const int c0 = (int)(((long long)P.H * mt) / gridDim.y), c1 = (int)(((long long)P.H * (mt + 1)) / gridDim.y);
      const int w = c1 - c0;
      for (int it = tid; it < cnt * w; it += kT5ConvThreads) {
        const int i = it / w, k = c0 + (it - i * w);
        const ActRow a = act_row<__nv_bfloat16>(P, sh.ca, pr, KIND, l, s_list[i]);
        P.h[(size_t)pr.prow[s_list[i]] * P.H + k] = a.f ? __ldcg(a.f + k) : WTraits<__nv_bfloat16>::load1(a.w, (size_t)k);
      }
    }
    // conversion share: tile row ci = tid / TPR, float4 chunks cs, cs + TPR, ... of each slab row
    // (cs = tid mod TPR: a warp reads whole 128-byte pieces of its rows)
    const int TPR = kT5ConvThreads / RB, ci = tid / TPR, cs = tid % TPR;
    const bool cv = ci < cnt;
    bool cbf = false;
    if (cv) cbf = act_row<__nv_bfloat16>(P, sh.ca, pr, KIND, l, s_list[ci]).f == nullptr;
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // own RoPE / gain copies
    asm volatile("bar.sync 2, %0;" ::"n"(kT5ConvThreads) : "memory");
    float ssq[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // per chunk column cs + TPR j of the row
    bool ok = true;
    for (int s = 0; s < slabs; ++s) {
      const int bs = s % kT5BStages;
      // slab s landed; the MMAs of slab s - kT5BStages (the B stage's last reader) completed
      const int sp = s - kT5BStages;
      if (!t5_wait(&sh.full[s % NST], (uint32_t)(s / NST) & 1u, abort, &P.ctl->status, P.wait_ns) ||
          !t5_wait(&sh.wfull[s % NST], (uint32_t)(s / NST) & 1u, abort, &P.ctl->status, P.wait_ns) ||
          (sp >= 0 && !t5_wait(&sh.empty[sp % NST], (uint32_t)(sp / NST) & 1u, abort, &P.ctl->status, P.wait_ns))) {
        ok = false;
        break;
      }
      if (cv) {
        const unsigned char* raw = rawb + (size_t)(s % NST) * RB * 256 + ci * 256;
        unsigned char* bst = bbase + (size_t)bs * RB * 256;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = cs + TPR * j;
          if (c >= 16) break;
          float x[4];
          if (cbf) {
            const uint2 w = *reinterpret_cast<const uint2*>(raw + c * 8);
            const float2 p0 = bf16x2_to_f2(w.x), p1 = bf16x2_to_f2(w.y);
            x[0] = p0.x; x[1] = p0.y; x[2] = p1.x; x[3] = p1.y;
          } else {
            const float4 v = *reinterpret_cast<const float4*>(raw + c * 16);
            x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) ssq[j] = fmaf(x[e], x[e], ssq[j]);
          if (kNormed) {
            const float4 g = *reinterpret_cast<const float4*>(s_gain + s * 64 + 4 * c);
            x[0] *= g.x; x[1] *= g.y; x[2] *= g.z; x[3] *= g.w;
          }
          uint2 hi, lo;
          t5_split(x[0], x[1], hi.x, lo.x);
          t5_split(x[2], x[3], hi.y, lo.y);
          *reinterpret_cast<uint2*>(bst + t5_swz(2 * ci, c >> 1) + (c & 1) * 8) = hi;
          *reinterpret_cast<uint2*>(bst + t5_swz(2 * ci + 1, c >> 1) + (c & 1) * 8) = lo;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the B slab visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.bfull[bs]);
    }
    // RMSNorm scales: a row's 16 chunk-column sums in column order (the same
    // order for every tile height); per-row offsets of the epilogue
    if (cv)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (cs + TPR * j < 16) s_ss[ci * 16 + cs + TPR * j] = ssq[j];
    if (tid < cnt) {
      const int gi = s_list[tid], r = pr.prow[gi], pos = pr.ppos[gi];
      long long e0, e1 = 0;
      if (KIND == kQKV) {
        const int slot = P.tree_n ? __ldcg(P.pslot + gi) : pos;                           // KV slot of the row
        e0 = (long long)r * P.nq * P.d;                                                     // q row
        e1 = ((((long long)(r / P.NS) * P.L + l) * 2) * P.GS + slot) * P.nkv * P.d;       // K row of the slot
      } else if (KIND == kO || KIND == kDown) {
        e0 = (long long)r * P.H;
      } else if (KIND == kGU) {
        e0 = (long long)r * P.F;
      } else {
        e0 = (long long)r * (1 + P.ND);
      }
      s_ep[3 * tid] = e0;
      s_ep[3 * tid + 1] = e1;
      s_ep[3 * tid + 2] = pos;
    }
    asm volatile("bar.sync 2, %0;" ::"n"(kT5ConvThreads) : "memory");
    if (tid < cnt) {
      float t = 0.0f;
      for (int c = 0; c < 16; ++c) t += s_ss[tid * 16 + c];
      s_inv[tid] = kNormed ? rsqrtf(t / (float)K + P.eps) : 1.0f;
    }
    if (ok && !t5_wait(&sh.dbar, 0, abort, &P.ctl->status, P.wait_ns)) ok = false;
    // one decision for all conversion warps (the epilogue's group barriers need all of them)
    int go = (ok && !*abort) ? 1 : 0;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n bar.red.and.pred q, 2, %2, p;\n selp.b32 %0, 1, 0, q;\n}"
                 : "=r"(go)
                 : "r"(go), "n"(kT5ConvThreads)
                 : "memory");
    if (go) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // epilogue: warp w reads TMEM lanes 32 (w mod 4) .. + 31 (weight rows) and
      // the column chunks (w / 4), (w / 4) + 2, ... of 16 columns (8 tile rows)
      const int m = 32 * (warp & 3) + lane;
      const bool second = kPair && m >= 64;          // pair kinds: A rows 64..127 hold the second rows
      const int mu = kPair ? (m & 63) : m;           // the row's unit within the tile
      const bool mvalid = mu < nun;
      float* xch = reinterpret_cast<float*>(smem + L.xch) + (warp >> 2) * 64 * 8;
      const float2* rope = rope_in_smem ? s_rope : P.rope;
      // per-lane constants of the weight row's unit
      const int uu = u0 + mu;
      int half = 0, hh = 0, e = 0;
      float* qkv_dst = nullptr;
      long long qkv_off = 0;
      if (KIND == kQKV) {
        half = P.d / 2;
        hh = uu / half;
        e = uu - hh * half;
        if (hh < P.nq) { qkv_dst = P.qbuf; qkv_off = (long long)hh * P.d + e; }
        else if (hh < P.nq + P.nkv) { qkv_dst = P.kv; qkv_off = (long long)(hh - P.nq) * P.d + e; }
        else { qkv_dst = P.kv; qkv_off = (long long)P.GS * P.nkv * P.d + (long long)(hh - P.nq - P.nkv) * P.d + e; }
      }
      int hv = 0, head = 0;
      if (KIND == kHeads) {
        const int hi = uu / P.V;
        hv = uu - hi * P.V;
        head = mvalid ? sh.heads[hi] : 0;
      }
      for (int ch = warp >> 2; ch < N / 16; ch += 2) {
        uint32_t v[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(16 * ch)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        float yv[8], pv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = 8 * ch + q;
          yv[q] = (__uint_as_float(v[2 * q]) + __uint_as_float(v[2 * q + 1])) * s_inv[i < cnt ? i : 0];
          pv[q] = 0.0f;
        }
        if (kPair) {
          // the second rows (warps 2, 3 of the group) hand their values to the first rows
          // (warps 0, 1): named barrier 3 + group among the group's four warps
          if (second)
#pragma unroll
            for (int q = 0; q < 8; ++q) xch[(m - 64) * 8 + q] = yv[q];
          asm volatile("bar.sync %0, 128;" ::"r"(3 + (warp >> 2)) : "memory");
          if (!second)
#pragma unroll
            for (int q = 0; q < 8; ++q) pv[q] = xch[m * 8 + q];
          asm volatile("bar.sync %0, 128;" ::"r"(3 + (warp >> 2)) : "memory");
          if (second) continue;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = 8 * ch + q;
          const int ii = i < cnt ? i : 0;
          const float y = yv[q];
          const float partner = pv[q];  // the other row of a pair
          if (i >= cnt || !mvalid) continue;
          const long long e0 = s_ep[3 * ii];
          if (KIND == kQKV) {
            const int pos = (int)s_ep[3 * ii + 2];
            const long long base = qkv_dst == P.qbuf ? e0 : s_ep[3 * ii + 1];
            float o0 = y, o1 = partner;
            if (hh < P.nq + P.nkv) {
              const float2 cs2 = rope[(size_t)pos * half + e];
              o0 = y * cs2.x - partner * cs2.y;
              o1 = partner * cs2.x + y * cs2.y;
            }
            qkv_dst[base + qkv_off] = o0;
            qkv_dst[base + qkv_off + half] = o1;
          } else if (KIND == kO || KIND == kDown) {
            float* hp = P.h + e0 + uu;
            *hp = __ldcg(hp) + y;
          } else if (KIND == kGU) {
            P.fbuf[e0 + uu] = y / (1.0f + expf(-y)) * partner;
          } else {
            const int pos = (int)s_ep[3 * ii + 2];
            const int slot = head - pos;
            float yy = y;
            if (slot >= 1 && slot <= P.KO) yy += __ldg(&P.otab[((size_t)(head - 1) * P.KO + slot - 1) * P.V + hv]);
            if (pos >= 1 && slot >= 0 && slot <= P.ND) P.logits[(e0 + slot) * P.V + hv] = yy;
          }
        }
      }
    }
  }
  // every role done: no copy in flight (copy warps waited), no MMA in flight
  // (the conversion warps or the MMA thread waited for the last commit)
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(N) : "memory");
  }
}

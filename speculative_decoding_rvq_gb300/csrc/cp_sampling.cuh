// cp_sampling.cuh -- logit processing, categorical draws and exact
// speculative acceptance, one warp per vocabulary row.
//
// Semantics ("Speculative Decoding, Beyond Text", section 02; "CodePredictor
// Speculative Decoding", "How a round works" step 3 and "Kernels"):
//  * processing: T == 0 -> one-hot argmax (lowest index on ties).  Else
//    z = fl32(logit / T); keep exactly min(k, V) entries by (z desc, index
//    asc) -- one MSB-first radix select over order-preserving keys, cost
//    independent of k; e_i = cp_expf(fl32(z_i - zmax)), S the sequential
//    float32 sum of the kept e_i in ascending index order, p_i = fl32(e_i / S).
//  * a processed row is a list (idx ascending, prob) of its support.
//  * categorical draw: sequential float32 prefix sums S_j over entries with
//    prob > 0 in index order; t = fl32(u * S_last); first j with S_j > t,
//    else the last candidate.
//  * acceptance: accept draft y iff u < fl32(p(y) / q(y)); at the first
//    rejection draw from max(0, p - q) (from p if that is all zero) and stop;
//    if all drafts are accepted and a bonus row exists, draw from it.
#pragma once
#include "cp_common.cuh"

namespace cpk {

// Load policies: data written by other CTAs of the same persistent launch is
// read through L2 only (ld.global.cg); shared-memory lists use plain loads.
struct LdCG {
  template <typename T> __device__ __forceinline__ static T ld(const T* p) { return __ldcg(p); }
};
struct LdPlain {
  template <typename T> __device__ __forceinline__ static T ld(const T* p) { return *p; }
};

// Stage a row of V floats from global into warp-private shared memory in
// one round trip: 16-byte async copies when the row is 16-byte aligned,
// batched scalar L2 loads for the tail or an unaligned row.
__device__ __forceinline__ void warp_stage_row(float* dst, const float* __restrict__ src, int V) {
  const int lane = threadIdx.x & 31;
  int done = 0;
  if ((((uintptr_t)src) & 15u) == 0) {
    done = V & ~3;
    warp_copy_async(dst, src, done * 4);
  }
  for (int i0 = done; i0 < V; i0 += 32 * 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + lane + 32 * j;
      v[j] = i < V ? __ldcg(src + i) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + lane + 32 * j;
      if (i < V) dst[i] = v[j];
    }
  }
  cp_async_wait_all();
  __syncwarp();
}

// Processes one row of V float32 logits, already staged in `keys`, with one
// warp.  keys: warp-private scratch of V uint32 holding the row (replaced by
// its keys); hist: warp-private 256 uint32; ebuf: warp-private min(k, V)
// floats; out_idx / out_prob: capacity min(k, V) (1 when T == 0).
// Returns the list length (all lanes).
static __device__ __noinline__ int warp_process_staged(uint32_t* keys, int V, int k, float T, uint32_t* hist,
                                                       float* ebuf, int* out_idx, float* out_prob) {
  const int lane = threadIdx.x & 31;
  float* row = reinterpret_cast<float*>(keys);
  if (T == 0.0f) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = lane; i < V; i += 32) {
      const float v = row[i];
      if (v > best || (v == best && i < bi)) { best = v; bi = i; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    if (lane == 0) { out_idx[0] = bi; out_prob[0] = 1.0f; }
    __syncwarp();
    return 1;
  }
  // keys of z = fl32(logit / T), in place; -0 is folded into +0 so ties match float compares
  uint32_t kmax = 0;
  for (int i = lane; i < V; i += 32) {
    float z = __fdiv_rn(row[i], T);
    if (z == 0.0f) z = 0.0f;
    const uint32_t key = float_key(z);
    keys[i] = key;
    kmax = max(kmax, key);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  __syncwarp();
  const int kk = k < V ? k : V;
  uint32_t prefix = 0, mask = 0;
  int need = kk;
  bool eq_all = (kk == V);
  for (int shift = 24; shift >= 0 && !eq_all; shift -= 8) {
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    for (int i = lane; i < V; i += 32) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane l owns bins 255-8l .. 248-8l (descending)
    uint32_t cnt[8];
    uint32_t chunk = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) { cnt[m] = hist[255 - 8 * lane - m]; chunk += cnt[m]; }
    uint32_t incl = chunk;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - chunk;
    const bool mine = excl < (uint32_t)need && (uint32_t)need <= incl;
    const uint32_t who = __ballot_sync(0xffffffffu, mine);
    const int src = __ffs(who) - 1;
    uint32_t bin = 0, above = 0, cbin = 0;
    if (mine) {
      uint32_t acc = excl;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        if (acc + cnt[m] >= (uint32_t)need) { bin = 255 - 8 * lane - m; above = acc; cbin = cnt[m]; break; }
        acc += cnt[m];
      }
    }
    bin = __shfl_sync(0xffffffffu, bin, src);
    above = __shfl_sync(0xffffffffu, above, src);
    cbin = __shfl_sync(0xffffffffu, cbin, src);
    need -= (int)above;
    prefix |= bin << shift;
    mask |= 0xFFu << shift;
    if ((int)cbin == need) eq_all = true;
    __syncwarp();
  }
  // compaction in ascending index order (strided layout: index = j*32 + lane);
  // each kept entry's e = cp_expf(z - zmax) is computed on the way
  const float zmax = key_float(kmax);
  int base = 0, eq_seen = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int j0 = 0; j0 < V; j0 += 32) {
    const int i = j0 + lane;
    bool sel = false, eq = false;
    uint32_t key = 0;
    if (i < V) {
      key = keys[i];
      const uint32_t km = key & mask;
      sel = km > prefix;
      eq = (km == prefix);
    }
    const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
    if (eq) sel = eq_all || (eq_seen + __popc(eqb & lt)) < need;
    eq_seen += __popc(eqb);
    const uint32_t selb = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const int pos = base + __popc(selb & lt);
      out_idx[pos] = i;
      ebuf[pos] = cp_expf(__fsub_rn(key_float(key), zmax));
    }
    base += __popc(selb);
  }
  __syncwarp();
  // softmax normalisation: sequential float32 sum in index order
  float S = 0.0f;
  if (lane == 0)
    for (int p = 0; p < kk; ++p) S = __fadd_rn(S, ebuf[p]);
  S = __shfl_sync(0xffffffffu, S, 0);
  for (int p = lane; p < kk; p += 32) out_prob[p] = __fdiv_rn(ebuf[p], S);
  __syncwarp();
  return kk;
}

// Stages one row of V float32 logits into `keys` and processes it (see
// warp_process_staged).
static __device__ __noinline__ int warp_process_row(const float* __restrict__ logits, int V, int k, float T,
                                                    uint32_t* keys, uint32_t* hist, float* ebuf, int* out_idx,
                                                    float* out_prob) {
  warp_stage_row(reinterpret_cast<float*>(keys), logits, V);
  return warp_process_staged(keys, V, k, T, hist, ebuf, out_idx, out_prob);
}

// ---- single-thread helpers (sequential float32 semantics) ----
template <typename LD = LdPlain>
__device__ __forceinline__ int list_sample(const int* idx, const float* prob, int n, float u) {
  float S = 0.0f;
  int last = -1;
  for (int j = 0; j < n; ++j) {
    const float pj = LD::ld(prob + j);
    if (pj > 0.0f) { S = __fadd_rn(S, pj); last = LD::ld(idx + j); }
  }
  if (last < 0) return -1;
  const float t = __fmul_rn(u, S);
  float acc = 0.0f;
  for (int j = 0; j < n; ++j) {
    const float pj = LD::ld(prob + j);
    if (!(pj > 0.0f)) continue;
    acc = __fadd_rn(acc, pj);
    if (acc > t) return LD::ld(idx + j);
  }
  return last;
}

template <typename LD = LdPlain>
__device__ __forceinline__ float list_lookup(const int* idx, const float* prob, int n, int y) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int v = LD::ld(idx + mid);
    if (v == y) return LD::ld(prob + mid);
    if (v < y) lo = mid + 1; else hi = mid - 1;
  }
  return 0.0f;
}

// Draw from max(0, p - q) over the union of two index-sorted lists.
// Returns -1 when the residual is zero everywhere.
template <typename LD = LdPlain>
__device__ __forceinline__ int residual_sample(const int* pi, const float* pp, int np, const int* qi,
                                               const float* qp, int nq, float u) {
  float S = 0.0f;
  int last = -1;
  for (int pass = 0; pass < 2; ++pass) {
    float t = 0.0f;
    if (pass == 1) {
      if (last < 0) return -1;
      t = __fmul_rn(u, S);
    }
    float acc = 0.0f;
    int a = 0, b = 0;
    while (a < np || b < nq) {
      const int ia = a < np ? LD::ld(pi + a) : 0x7fffffff;
      const int ib = b < nq ? LD::ld(qi + b) : 0x7fffffff;
      int i;
      float pv = 0.0f, qv = 0.0f;
      if (ia <= ib) { i = ia; pv = LD::ld(pp + a); ++a; if (ib == ia) { qv = LD::ld(qp + b); ++b; } }
      else { i = ib; qv = LD::ld(qp + b); ++b; }
      const float d = __fsub_rn(pv, qv);
      const float r = d > 0.0f ? d : 0.0f;
      if (!(r > 0.0f)) continue;
      if (pass == 0) { S = __fadd_rn(S, r); last = i; }
      else {
        acc = __fadd_rn(acc, r);
        if (acc > t) return i;
      }
    }
    if (pass == 1) return last;
  }
  return last;
}

}  // namespace cpk

namespace cpk {

// ---- dense-row variants (probability-input mode): same sequential orders ----
__device__ __forceinline__ int dense_sample(const float* __restrict__ w, int V, float u) {
  float S = 0.0f;
  int last = -1;
  for (int i = 0; i < V; ++i) {
    const float v = __ldg(w + i);
    if (v > 0.0f) { S = __fadd_rn(S, v); last = i; }
  }
  if (last < 0) return -1;
  const float t = __fmul_rn(u, S);
  float acc = 0.0f;
  for (int i = 0; i < V; ++i) {
    const float v = __ldg(w + i);
    if (!(v > 0.0f)) continue;
    acc = __fadd_rn(acc, v);
    if (acc > t) return i;
  }
  return last;
}

__device__ __forceinline__ int dense_residual(const float* __restrict__ p, const float* __restrict__ q, int V,
                                              float u) {
  float S = 0.0f;
  int last = -1;
  for (int i = 0; i < V; ++i) {
    const float d = __fsub_rn(__ldg(p + i), __ldg(q + i));
    if (d > 0.0f) { S = __fadd_rn(S, d); last = i; }
  }
  if (last < 0) return -1;
  const float t = __fmul_rn(u, S);
  float acc = 0.0f;
  for (int i = 0; i < V; ++i) {
    const float d = __fsub_rn(__ldg(p + i), __ldg(q + i));
    if (!(d > 0.0f)) continue;
    acc = __fadd_rn(acc, d);
    if (acc > t) return i;
  }
  return last;
}

}  // namespace cpk

// Device helpers shared by the frame-loop kernels: bounded waits that honour
// a grid-wide abort flag, counter atomics with explicit memory order, f16
// packing, and the per-warp RMSNorm + RoPE and score reduction of attention.
// A params type passed to the waits has int* members abort_flag and status
// and a long long spin_limit (clock64 ticks).
#pragma once

#include "qp_common.cuh"
#include "qp_internal.h"
#include "qp_ptx.cuh"

namespace qp {
namespace {

// ------------------------------------------------------------------ waits
template <class Par>
__device__ __forceinline__ void abort_all(const Par& p) {
  set_status(p.status, QP_ERR_TIMEOUT);
  atomicExch(p.abort_flag, 1);
}
template <class Par>
__device__ __forceinline__ bool aborted(const Par& p) { return *(volatile int*)p.abort_flag != 0; }

// Until *ctr >= want (acquire), bounded.  After two misses each poll is
// spaced by a short sleep, which eases the load the waiting threads of every
// CTA put on the counters' L2 lines (about 1 % per step, measured).
template <class Par>
__device__ bool poll_geq(const Par& p, const unsigned* ctr, unsigned want) {
  if (ld_acquire_u32(ctr) >= want) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (ld_acquire_u32(ctr) >= want) return true;
    if (it > 2) __nanosleep(32);
    if ((it & 63) == 0) {
      if (aborted(p)) return false;
      if (clock64() - t0 > p.spin_limit) { abort_all(p); return false; }
    }
  }
}

// mbarrier phase wait, bounded, abandoning when the grid aborts.
template <class Par>
__device__ bool mwait(const Par& p, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255) == 0) {
      if (aborted(p)) return false;
      if (clock64() - t0 > p.spin_limit) { abort_all(p); return false; }
    }
  }
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A relaxed add: after fence_acq_rel_gpu(), a run of these releases the
// writes before the fence as each red.release would, with one fence.
__device__ __forceinline__ void red_relaxed_add(unsigned* p, unsigned v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Fetch-and-add with acquire-release semantics at GPU scope: publishes this
// CTA's earlier writes (ordered before it by bar.sync) and, for the caller
// that completes a count, makes every earlier contributor's writes visible.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// ------------------------------------------------------ f16 operand range
// A GEMM operand row built from the residual stream (or from H) is
// multiplied by 2^-e before its f16 conversion, and the GEMM's f32 result
// by 2^e after it (both exact), so that rows of any magnitude stay inside
// f16's range (65504).  e comes from the mean square ms of a reference row
// known before the operand is built -- the row itself where it is complete,
// else the same frame's most recent complete residual row: 2^-e brings that
// row's RMS into [2^-5, 2^-4), or e = 0 (no scaling) when the RMS is below
// 2^-5.  A row may grow far past its reference within one sublayer before
// 2^-e * |x| * |w_norm| reaches 65504, and f16's relative precision does not
// depend on the scale above its smallest normal value (2^-14).
__device__ __forceinline__ int range_exp(float ms) {
  const int E = int((__float_as_uint(ms) >> 23) & 255u) - 127;   // floor(log2(ms)) for ms >= 2^-126
  const int e = (E >> 1) + 5;                                      // floor(log2(RMS)) + 5
  return e < 0 ? 0 : (e > 100 ? 100 : e);
}
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(uint32_t(127 + e) << 23); }   // |e| <= 126

__device__ __forceinline__ uint2 pack4_f16(float a, float b, float c, float d) {
  return make_uint2(uint32_t(f32_to_f16_bits(a)) | (uint32_t(f32_to_f16_bits(b)) << 16),
                    uint32_t(f32_to_f16_bits(c)) | (uint32_t(f32_to_f16_bits(d)) << 16));
}
__device__ __forceinline__ float4 unpack4_f16(uint2 v) {
  return make_float4(f16_bits_to_f32(v.x & 0xffff), f16_bits_to_f32(v.x >> 16), f16_bits_to_f32(v.y & 0xffff),
                     f16_bits_to_f32(v.y >> 16));
}


// RMSNorm of a 128-vector held as 4 values per lane, then rotate-half RoPE
// at position pos (pairs (i, i+64) sit in lanes l and l^16).
__device__ __forceinline__ float4 norm_rope(float4 x, const float* nw, float eps, const float2* cs, int lane) {
  const float ss = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
  const float r = rsqrtf(ss / 128.f + eps);
  const float4 w = *reinterpret_cast<const float4*>(nw + lane * 4);
  float v[4] = {x.x * r * w.x, x.y * r * w.y, x.z * r * w.z, x.w * r * w.w};
  float o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float partner = __shfl_xor_sync(0xffffffffu, v[e], 16);
    const float2 c = cs[(lane * 4 + e) & 63];
    o[e] = lane < 16 ? v[e] * c.x - partner * c.y : v[e] * c.x + partner * c.y;
  }
  return make_float4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// ------------------------------------------------------ top-k selection
// Shared memory one group of threads needs for one frame's decision.
struct TopkScratch {
  unsigned cnt[2][4];          // per round parity, warp: counts of the digits 1, 2, 3 (10 bits each), or of ties
  int wtot[4];                 // per-warp totals of the tie scan
  int last_tie;                // index of the last kept key equal to the threshold
  unsigned long long red[4];   // per-warp (value, index) maxima
  float rsum[4];               // per-warp partial sums (row scale)
};

// Exclusive prefix sum of v over the NG threads of a group in thread order
// (tg = thread index in the group; wtot holds NG / 32 ints; `bar` is the
// group's named barrier).  Ends with the barrier that publishes the warp
// totals; the group's next barrier must come before wtot is rewritten.
template <int NG>
__device__ int group_exclusive_scan(int v, int* wtot, int bar, int tg) {
  const int lane = tg & 31, warp = tg >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wtot[warp] = incl;
  named_bar(bar, NG);
  int off = 0;
  for (int w = 0; w < warp; ++w) off += wtot[w];
  return off + incl - v;
}

// The Gumbel top-k decision of one frame by a group of NG = 128 threads (tg
// = the thread's index in the group, `bar` the group's named barrier): z =
// logit * rs / T; the candidate set is the top_k largest z, ties at the
// threshold kept lowest index first; the code is the argmax over the set of
// z + g, lowest index on ties.  Every thread of the group returns it.  V is
// a multiple of NG and at most 32 * NG; keys (shared memory, V words) is
// read only when ties at the threshold must be ranked.
//
// The top_k-th largest order key comes from a bitwise radix select with no
// atomics and no divergent branches: each thread holds its keys (indices tg
// + NG u) in registers, and each of 16 rounds fixes two more bits of the
// threshold from the counts of the keys sharing the bits fixed so far whose
// next two bits are 1, 2 or 3 -- packed 10 bits apart into one word, summed
// over the warp by one reduction, then one group barrier (the count buffers
// alternate by round, so a round needs no second barrier).
template <int NG>
__device__ int gumbel_topk_group(const float* l, float rs, float T, const float* gb, int V, int top_k,
                                 uint32_t* keys, TopkScratch& sc, int bar, int tg) {
  static_assert(NG == 128, "four warps per group");
  constexpr int KPT = 32;   // keys per thread at most (V <= 4096)
  const int lane = tg & 31, w = tg >> 5, kpt = V / NG;
  uint32_t key[KPT];
#pragma unroll
  for (int u0 = 0; u0 < KPT; u0 += 8) {   // eight loads in flight at a time
    float lv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) lv[u] = u0 + u < kpt ? __ldcg(l + tg + (u0 + u) * NG) : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) key[u0 + u] = u0 + u < kpt ? f32_order_key(lv[u] * rs / T) : 0u;
  }
  uint32_t prefix = 0;
  int rem = top_k, par = 0;
  for (int shift = 30; shift >= 0; shift -= 2, par ^= 1) {
    const uint32_t hmask = shift == 30 ? 0u : (0xFFFFFFFFu << (shift + 2));
    unsigned packed = 0;   // digit d >= 1 counts at bits 10 (d - 1): a warp's count is at most 1024 - 1
#pragma unroll
    for (int u = 0; u < KPT; ++u) {
      if (u >= kpt) break;   // warp-uniform
      const uint32_t kk = key[u], d = (kk >> shift) & 3u;
      const unsigned one = (kk & hmask) == prefix && d != 0u ? 1u : 0u;
      packed += one << (10u * (d - 1u) & 31u);
    }
    packed = __reduce_add_sync(0xffffffffu, packed);
    if (lane == 0) sc.cnt[par][w] = packed;
    named_bar(bar, NG);
    int s1 = 0, s2 = 0, s3 = 0;
#pragma unroll
    for (int i = 0; i < NG / 32; ++i) {
      const unsigned c = sc.cnt[par][i];
      s1 += int(c & 1023u); s2 += int((c >> 10) & 1023u); s3 += int(c >> 20);
    }
    uint32_t d;
    if (s3 >= rem) d = 3u;
    else if (s3 + s2 >= rem) { d = 2u; rem -= s3; }
    else if (s3 + s2 + s1 >= rem) { d = 1u; rem -= s3 + s2; }
    else { d = 0u; rem -= s3 + s2 + s1; }
    prefix |= d << shift;
  }
  const uint32_t kth = prefix;   // the top_k-th largest key; rem of the keys equal to it are kept
  unsigned eq = 0;
#pragma unroll
  for (int u = 0; u < KPT; ++u) {
    if (u >= kpt) break;
    eq += key[u] == kth ? 1u : 0u;
  }
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) sc.cnt[par][w] = eq;
  named_bar(bar, NG);
  int equal = 0;
#pragma unroll
  for (int i = 0; i < NG / 32; ++i) equal += int(sc.cnt[par][i]);
  int last_tie = V;
  if (rem < equal) {   // not every key equal to the threshold is kept: the rem lowest indices are
#pragma unroll
    for (int u = 0; u < KPT; ++u)
      if (u < kpt) keys[tg + u * NG] = key[u];
    named_bar(bar, NG);
    const int lo = tg * kpt;
    int cnt = 0;
    for (int i = lo; i < lo + kpt; ++i) cnt += keys[i] == kth;
    int rank = group_exclusive_scan<NG>(cnt, sc.wtot, bar, tg);
    if (rank < rem && rem <= rank + cnt)
      for (int i = lo; i < lo + kpt; ++i)
        if (keys[i] == kth && ++rank == rem) { sc.last_tie = i; break; }
    named_bar(bar, NG);
    last_tie = sc.last_tie;
  }
  // the kept keys' logits and noise: predicated loads, all in flight together
  unsigned long long best = 0ull;
#pragma unroll
  for (int u0 = 0; u0 < KPT; u0 += 16) {
    if (u0 >= kpt) break;
    float lz[16], gz[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = tg + (u0 + u) * NG;
      const bool in = u0 + u < kpt && (key[u0 + u] > kth || (key[u0 + u] == kth && i <= last_tie));
      lz[u] = in ? __ldcg(l + i) : 0.f;
      gz[u] = in ? __ldg(gb + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = tg + (u0 + u) * NG;
      const bool in = u0 + u < kpt && (key[u0 + u] > kth || (key[u0 + u] == kth && i <= last_tie));
      const unsigned long long pk = in ? pack_argmax(lz[u] * rs / T + gz[u], i) : 0ull;
      best = pk > best ? pk : best;
    }
  }
  best = warp_max_u64(best);
  if (lane == 0) sc.red[w] = best;
  named_bar(bar, NG);
  unsigned long long v = sc.red[0];
#pragma unroll
  for (int i = 1; i < NG / 32; ++i) v = sc.red[i] > v ? sc.red[i] : v;
  return unpack_argmax_index(v);
}

// Sixteen warp-wide sums: lane l ends with the total over all 32 lanes of
// v[(l >> 1) & 15] (lanes 2i and 2i + 1 both hold sum i).  Four halving
// exchanges, then the lane pairs meet.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int o = 16; o >= 2; o >>= 1) {
    const int c = o >> 1;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < c; ++i) {
      const float send = upper ? v[i] : v[i + c];
      const float keep = upper ? v[i + c] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

}  // namespace
}  // namespace qp

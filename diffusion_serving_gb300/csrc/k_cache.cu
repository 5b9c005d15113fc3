// Cache bookkeeping and slot writes.
//
//  * k_advance   slot reservation for the next chunk (flashdreams issue "add an opt-in
//                circular KV policy for streaming attention", "proposed boundary":
//                reservation is separate from writes and lives in device memory).
//  * k_reset     row lifecycle reset (same section).
//  * k_set_lengths  active prefix kv_len (fish-speech PR "pass only active KV cache
//                prefix to SDPA", "Change") and packed offsets cu_seqlens (TensorRT-LLM
//                PR "FA4 variable-length cross-attention", Description).
//  * k_write     index_copy-style row scatter (lingbot-world PR "refactor(kv):
//                index_copy_ for KV-cache writes", Summary): bytes copied unchanged in
//                16-byte vectors, slot taken from device memory so replays of a
//                captured graph write the slot the device holds.
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace {

__global__ void k_advance(int32_t* __restrict__ meta, int B, int row, int n, int layout, int sink,
                          int window, int chunk, int cap) {
  kvc_pdl_wait();
  kvc_pdl_release();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    if (row >= 0 && b != row) continue;
    int32_t* r = meta + kvc_meta_row(b);
    const int k = r[KVC_ROW_CHUNKS];
    if (layout == KVC_CIRCULAR) {
      const int64_t first = (int64_t)k * chunk;
      int base;
      if (first < window) {
        base = (int)first;                               // still filling
      } else {
        const int roll = (window - sink) / chunk;        // rolling chunks
        const int64_t idx = ((int64_t)k - sink / chunk) % roll;
        base = sink + (int)idx * chunk;                  // oldest rolling chunk
      }
      const int64_t filled = first + chunk < window ? first + chunk : window;
      r[KVC_ROW_CHUNKS] = k + 1;
      r[KVC_ROW_BASE] = base;
      r[KVC_ROW_FILLED] = (int)filled;
      r[KVC_ROW_KVLEN] = (int)filled;
    } else {  // LINEAR
      const int filled = r[KVC_ROW_FILLED];
      if ((int64_t)filled + n > cap) {
        atomicOr(meta + KVC_META_ERR, KVC_DEV_OVERFLOW);
        continue;
      }
      r[KVC_ROW_CHUNKS] = k + 1;
      r[KVC_ROW_BASE] = filled;
      r[KVC_ROW_FILLED] = filled + n;
      r[KVC_ROW_KVLEN] = filled + n;
    }
  }
}

__global__ void k_reset(int32_t* __restrict__ meta, int B, int row) {
  kvc_pdl_wait();
  kvc_pdl_release();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    if (row >= 0 && b != row) continue;
    int32_t* r = meta + kvc_meta_row(b);
    r[KVC_ROW_CHUNKS] = 0;
    r[KVC_ROW_BASE] = 0;
    r[KVC_ROW_FILLED] = 0;
    r[KVC_ROW_KVLEN] = 0;
  }
}

__global__ void k_set_lengths(int32_t* __restrict__ meta, int B, int cap, const int32_t* __restrict__ kv_len,
                              const int32_t* __restrict__ cu) {
  __shared__ int ok;
  kvc_pdl_wait();
  kvc_pdl_release();
  if (kv_len != nullptr) {
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      const int n = kv_len[b];
      if (n < 1 || n > cap) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_KVLEN);
      else meta[kvc_meta_row(b) + KVC_ROW_KVLEN] = n;
    }
  }
  if (cu == nullptr) return;
  if (threadIdx.x == 0) {
    int good = cu[0] == 0;
    for (int b = 0; b < B && good; ++b) good = cu[b + 1] > cu[b];
    good = good && cu[B] <= cap;
    ok = good;
    if (!good) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_CUSEQ);
  }
  __syncthreads();
  if (!ok) return;
  for (int b = threadIdx.x; b <= B; b += blockDim.x) meta[kvc_meta_cu(B) + b] = cu[b];
  for (int b = threadIdx.x; b < B; b += blockDim.x) meta[kvc_meta_row(b) + KVC_ROW_KVLEN] = cu[b + 1] - cu[b];
}

// One warp per (tensor, row b, token i): the warp resolves the destination row once,
// then its lanes copy the row's 16-byte vectors, 4 loads in flight per lane before
// the stores.  Destination row of (b, i):
//   slots given:  b * cap + slots[i]
//   reserved:     b * cap + base_b + i      (LINEAR also requires base_b + i < filled_b)
//   packed:       cu[b] + i for i < len_b (later tokens are padding and are skipped)
constexpr int kWriteThreads = 256;
constexpr int kWriteUnroll = 4;

__global__ void __launch_bounds__(kWriteThreads)
k_write(const uint4* __restrict__ ksrc, const uint4* __restrict__ vsrc, uint4* __restrict__ kdst,
        uint4* __restrict__ vdst, int32_t* __restrict__ meta, const int32_t* __restrict__ lens,
        const int32_t* __restrict__ slots, int B, int n, int row_vecs, int cap, int layout) {
  kvc_pdl_wait();
  kvc_pdl_release();
  const int lane = threadIdx.x & 31;
  const int rows_per_tensor = B * n;
  const int rows = 2 * rows_per_tensor;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const int t = r >= rows_per_tensor;
    const int e = r - (t ? rows_per_tensor : 0);
    const int b = e / n;
    const int i = e - b * n;
    int64_t drow = -1;
    if (layout == KVC_PACKED) {
      const int32_t* cu = lens + kvc_meta_cu(B);
      const int lo = cu[b], hi = cu[b + 1];
      if (i < hi - lo && lo >= 0 && hi <= cap) drow = lo + i;
    } else if (slots != nullptr) {
      const int s = slots[i];
      if (s >= 0 && s < cap) drow = (int64_t)b * cap + s;
      else if (lane == 0 && t == 0) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_SLOT);
    } else {
      const int32_t* m = meta + kvc_meta_row(b);
      const int chunks = m[KVC_ROW_CHUNKS];
      const int s = m[KVC_ROW_BASE] + i;
      const bool ok = chunks > 0 && s >= 0 && s < cap && (layout != KVC_LINEAR || s < m[KVC_ROW_FILLED]);
      if (ok) drow = (int64_t)b * cap + s;
      else if (lane == 0 && t == 0) atomicOr(meta + KVC_META_ERR, chunks > 0 ? KVC_DEV_BAD_SLOT : KVC_DEV_NO_CHUNK);
    }
    if (drow < 0) continue;
    const uint4* src = (t ? vsrc : ksrc) + (int64_t)e * row_vecs;
    uint4* dst = (t ? vdst : kdst) + drow * row_vecs;
    for (int v0 = lane; v0 < row_vecs; v0 += 32 * kWriteUnroll) {
      uint4 val[kWriteUnroll];
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < row_vecs) val[u] = __ldg(src + v);
      }
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < row_vecs) dst[v] = val[u];
      }
    }
  }
}

// Write with RoPE fused into the K half: K rows are rotated at their absolute position
// before they are stored, V rows are copied unchanged (flashdreams issue "add an opt-in
// circular KV policy for streaming attention", "proposed boundary": absolute positions
// determine RoPE before storage).  Pair j of a head, (x[2j], x[2j+1]), turns by the
// angle whose (cos, sin) the caller's table holds at [pos][j]:
//   (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos),
// and the store receives the exact value of each component rounded once to nearest-even
// in the store type (finite inputs).
// Absolute position of token i: CIRCULAR (chunks - 1) * chunk + i; LINEAR base + i, or
// slots[i] when slots are given; PACKED i.  Rows whose position is outside the table
// are skipped and set KVC_DEV_BAD_POS.
//
// Rounding once, 16-bit stores.  Component a*b - c*d (a, c of the store type, exact in
// fp32; b, d fp32 table entries; the second component x0 sin + x1 cos is x0*sin -
// x1*(-cos)).  Fast path, in fp32 (two components per packed fp32x2 instruction):
//   q = c*d, its error eq = fma(c, d, -q) (exact while |c*d| >= 2^-100, or zero when c or
//   d is), r = fma(a, b, -q), r2 = r - eq.
// Then |r2 - (a*b - c*d)| <= half an ulp of r2 plus half an ulp of r; with
// |q| <= 2^20 |r2| (no deep cancellation) r is within a binade of r2, so the error is at
// most 1.5 ulp of r2.  Rounding r2 gives the answer unless r2 lies within 2 fp32 ulps of a
// rounding midpoint of the store type, which its low bits show (16 of them for bf16, 13
// for fp16 normal values).  Every other element (a fraction of a percent with N(0, 1)
// data, plus fp16 subnormal results) takes the exact path: in fp64 the products are exact
// (<= 35 significant bits), hi = fl(a*b - c*d) with its exact rest (Knuth's TwoSum), and
// hi + rest is rounded to fp32 by round-to-odd (truncate, then set the last bit when
// inexact), which has enough spare bits for one correct rounding to the store type.
__device__ __forceinline__ void kvc_two_sum(double a, double b, double& s, double& e) {
  s = a + b;
  const double bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// a*b - c*d rounded to fp32 by round-to-odd.
__device__ __noinline__ float kvc_rot_odd(float a, float b, float c, float d) {
  double hi, rest;
  kvc_two_sum((double)a * (double)b, -((double)c * (double)d), hi, rest);
  const float t = __double2float_rz(hi);
  uint32_t u = __float_as_uint(t);
  if ((double)t == hi) {
    if (rest == 0.0) return t;                       // exact
    if ((rest > 0.0) != (hi > 0.0)) u -= 1;          // the exact value is just inside t
  }
  return __uint_as_float(u | 1u);
}

template <typename T> struct Round16;
template <> struct Round16<__nv_bfloat16> {
  using T2 = __nv_bfloat162;
  __device__ static float2 unpack(T2 h) { return __bfloat1622float2(h); }
  __device__ static T2 pack(float a, float b) { return __floats2bfloat162_rn(a, b); }
  __device__ static __nv_bfloat16 rn(float x) { return __float2bfloat16_rn(x); }
  // r2 is more than 2 fp32 ulps away from every bf16 rounding midpoint
  __device__ static bool clear(float r2) { return (__float_as_uint(r2) & 0xFFFFu) - 0x7FFEu > 4u; }
};
template <> struct Round16<__half> {
  using T2 = __half2;
  __device__ static float2 unpack(T2 h) { return __half22float2(h); }
  __device__ static T2 pack(float a, float b) { return __floats2half2_rn(a, b); }
  __device__ static __half rn(float x) { return __float2half_rn(x); }
  __device__ static bool clear(float r2) {
    const float m = fabsf(r2);
    if (m >= 65536.f) return true;                   // every such value rounds to infinity
    return m >= 0x1p-14f && (__float_as_uint(r2) & 0x1FFFu) - 0x0FFEu > 4u;
  }
};

// Per-lane constants of one pair: (cos, sin), (sin, -cos), (-sin, cos).
struct RopePair {
  float2 cs, sc, nsc;
};

template <typename T> struct Pack;
template <typename T> struct Pack16 {
  using R = Round16<T>;
  static constexpr int kPairs = 4;   // pairs per 16-byte vector
  __device__ static void rot(uint4& u, const RopePair* cp) {
    typename R::T2* h = reinterpret_cast<typename R::T2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = R::unpack(h[i]);
      const float2 x1 = make_float2(x.y, x.y);
      const float2 nq = __fmul2_rn(x1, cp[i].nsc);                          // -q
      const float2 eq = __ffma2_rn(x1, cp[i].sc, nq);                       // exact error of q
      const float2 r = __ffma2_rn(make_float2(x.x, x.x), cp[i].cs, nq);
      const float2 r2 = __ffma2_rn(eq, make_float2(-1.f, -1.f), r);         // r - eq
      const float qa = fabsf(nq.x), qb = fabsf(nq.y);
      const bool ok_a = ((qa >= 0x1p-100f && qa <= fabsf(r2.x) * 0x1p20f) ||
                         (qa == 0.f && (x.y == 0.f || cp[i].sc.x == 0.f))) && R::clear(r2.x);
      const bool ok_b = ((qb >= 0x1p-100f && qb <= fabsf(r2.y) * 0x1p20f) ||
                         (qb == 0.f && (x.y == 0.f || cp[i].sc.y == 0.f))) && R::clear(r2.y);
      if (ok_a && ok_b) {
        h[i] = R::pack(r2.x, r2.y);
      } else {
        const float a = ok_a ? r2.x : kvc_rot_odd(x.x, cp[i].cs.x, x.y, cp[i].sc.x);
        const float b = ok_b ? r2.y : kvc_rot_odd(x.x, cp[i].cs.y, x.y, cp[i].sc.y);
        h[i] = R::pack(a, b);   // r2 itself where it was clear, the odd-rounded value elsewhere
      }
    }
  }
};
template <> struct Pack<__nv_bfloat16> : Pack16<__nv_bfloat16> {};
template <> struct Pack<__half> : Pack16<__half> {};
// fp32 stores: the products (<= 48 significant bits) are exact in fp64; hi = fl(a*b - c*d)
// with its exact rest (TwoSum).  Rounding hi to fp32 is the answer unless hi sits exactly
// on an fp32 midpoint with a non-zero rest, in which case the rest's sign picks the side.
__device__ __forceinline__ float kvc_rot_round_f32(float a, float b, float c, float d) {
  double hi, rest;
  kvc_two_sum((double)a * (double)b, -((double)c * (double)d), hi, rest);
  const float f = __double2float_rn(hi);
  if (rest == 0.0) return f;
  const float lo_f = __double2float_rd(hi), hi_f = __double2float_ru(hi);
  if (lo_f == hi_f) return f;
  const double up = isinf(hi_f) ? copysign(0x1p128, (double)hi_f) : (double)hi_f;
  const double down = isinf(lo_f) ? copysign(0x1p128, (double)lo_f) : (double)lo_f;
  if (hi != 0.5 * (up + down)) return f;
  return rest > 0.0 ? hi_f : lo_f;
}
template <> struct Pack<float> {
  static constexpr int kPairs = 2;
  __device__ static void rot(uint4& u, const RopePair* cp) {
    float* f = reinterpret_cast<float*>(&u);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float x0 = f[2 * i], x1 = f[2 * i + 1];
      f[2 * i] = kvc_rot_round_f32(x0, cp[i].cs.x, x1, cp[i].sc.x);
      f[2 * i + 1] = kvc_rot_round_f32(x0, cp[i].cs.y, x1, cp[i].sc.y);
    }
  }
};

// One warp per token (b, i): it resolves the destination row and the position once, then
// its lanes load the token's K and V vectors together (V is stored as it came, K after
// the rotation), so the copy of V keeps memory busy while K is rotated.
template <typename T>
__global__ void __launch_bounds__(kWriteThreads)
k_write_rope(const uint4* __restrict__ ksrc, const uint4* __restrict__ vsrc, uint4* __restrict__ kdst,
             uint4* __restrict__ vdst, int32_t* __restrict__ meta, const int32_t* __restrict__ lens,
             const int32_t* __restrict__ slots, const float2* __restrict__ rope, int rope_positions, int B, int n,
             int row_vecs, int cap, int layout, int chunk, int head_dim) {
  constexpr int P = Pack<T>::kPairs;
  constexpr int U = 3;                    // vectors of K (and of V) in flight per lane
  kvc_pdl_wait();
  kvc_pdl_release();
  const int lane = threadIdx.x & 31;
  const int tokens = B * n;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int half_d = head_dim / 2;
  for (int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; e < tokens; e += warps) {
    const int b = e / n;
    const int i = e - b * n;
    int64_t drow = -1;
    int pos = -1;
    if (layout == KVC_PACKED) {
      const int32_t* cu = lens + kvc_meta_cu(B);
      const int lo = cu[b], hi = cu[b + 1];
      if (i < hi - lo && lo >= 0 && hi <= cap) drow = lo + i;
      pos = i;
    } else if (slots != nullptr) {
      const int sl = slots[i];
      if (sl >= 0 && sl < cap) drow = (int64_t)b * cap + sl;
      else if (lane == 0) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_SLOT);
      pos = sl;
    } else {
      const int32_t* m = meta + kvc_meta_row(b);
      const int chunks = m[KVC_ROW_CHUNKS];
      const int sl = m[KVC_ROW_BASE] + i;
      const bool ok = chunks > 0 && sl >= 0 && sl < cap && (layout != KVC_LINEAR || sl < m[KVC_ROW_FILLED]);
      if (ok) drow = (int64_t)b * cap + sl;
      else if (lane == 0) atomicOr(meta + KVC_META_ERR, chunks > 0 ? KVC_DEV_BAD_SLOT : KVC_DEV_NO_CHUNK);
      pos = layout == KVC_CIRCULAR ? (chunks - 1) * chunk + i : sl;
    }
    if (drow < 0) continue;
    if (pos < 0 || pos >= rope_positions) {        // neither K nor V of such a token is written
      if (lane == 0) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_POS);
      continue;
    }
    // A lane's vectors v, v + 32, ... all start at the same pair of their head: 32
    // vectors of P pairs span whole heads (head_dim / 2 is 32 or 64 pairs), so the
    // lane's (cos, sin) entries are read once per token.
    RopePair cp[P];
    {
      const float2* cs_row = rope + (int64_t)pos * half_d + (lane * P) % half_d;
#pragma unroll
      for (int k = 0; k < P; ++k) {
        const float2 t = __ldg(cs_row + k);
        cp[k].cs = t;
        cp[k].sc = make_float2(t.y, -t.x);
        cp[k].nsc = make_float2(-t.y, t.x);
      }
    }
    const uint4* ks = ksrc + (int64_t)e * row_vecs;
    const uint4* vs = vsrc + (int64_t)e * row_vecs;
    uint4* kd = kdst + drow * row_vecs;
    uint4* vd = vdst + drow * row_vecs;
    for (int v0 = lane; v0 < row_vecs; v0 += 32 * U) {
      uint4 kv[U], vv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (v0 + 32 * u < row_vecs) {
          kv[u] = __ldg(ks + v0 + 32 * u);
          vv[u] = __ldg(vs + v0 + 32 * u);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (v0 + 32 * u < row_vecs) vd[v0 + 32 * u] = vv[u];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (v0 + 32 * u < row_vecs) {
          Pack<T>::rot(kv[u], cp);
          kd[v0 + 32 * u] = kv[u];
        }
      }
    }
  }
}

// Append to a LINEAR store in one launch: kvc_advance(row -1, n) and the write of the
// reserved chunk together, for a decode step's few tokens (the fish-speech PR "pass only
// active KV cache prefix to SDPA", "Change": decode step i stores its token at T + i and
// attends T + i + 1 slots).  One block: every row's fill count is read first, the rows
// are copied to slots filled_b + i, and only then is the meta block advanced, so no warp
// reads a count another has already moved.  A row that would pass its capacity sets
// KVC_DEV_OVERFLOW and is left unchanged, as kvc_advance does.
constexpr int kAppendMaxRows = 1024;

__global__ void __launch_bounds__(kWriteThreads)
k_append(const uint4* __restrict__ ksrc, const uint4* __restrict__ vsrc, uint4* __restrict__ kdst,
         uint4* __restrict__ vdst, int32_t* __restrict__ meta, int B, int n, int row_vecs, int cap) {
  __shared__ int s_base[kAppendMaxRows];
  kvc_pdl_wait();
  kvc_pdl_release();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int filled = meta[kvc_meta_row(b) + KVC_ROW_FILLED];
    const bool ok = filled >= 0 && (int64_t)filled + n <= cap;
    if (!ok) atomicOr(meta + KVC_META_ERR, KVC_DEV_OVERFLOW);
    s_base[b] = ok ? filled : -1;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int rows = 2 * B * n;
  for (int r = threadIdx.x >> 5; r < rows; r += blockDim.x >> 5) {
    const int t = r >= B * n;
    const int e = r - (t ? B * n : 0);
    const int b = e / n, i = e - b * n;
    if (s_base[b] < 0) continue;
    const uint4* src = (t ? vsrc : ksrc) + (int64_t)e * row_vecs;
    uint4* dst = (t ? vdst : kdst) + ((int64_t)b * cap + s_base[b] + i) * row_vecs;
    for (int v = lane; v < row_vecs; v += 32) dst[v] = __ldg(src + v);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    if (s_base[b] < 0) continue;
    int32_t* m = meta + kvc_meta_row(b);
    m[KVC_ROW_CHUNKS] += 1;
    m[KVC_ROW_BASE] = s_base[b];
    m[KVC_ROW_FILLED] = s_base[b] + n;
    m[KVC_ROW_KVLEN] = s_base[b] + n;
  }
}

// Comparator for measurement, not on the path: the copy a chronological sink + window
// store makes once per chunk step (flashdreams issue "add an opt-in circular KV policy
// for streaming attention", "current path": the retained keys and values are cloned and
// copied back one chunk to the left).  Rows [first, first + count) of every batch row
// move between `src` (row stride src_cap) and `dst` (row stride dst_cap), K and V in
// one launch; the roll is two such launches: store -> scratch, scratch -> store.
__global__ void __launch_bounds__(kWriteThreads)
k_copy_rows(const uint4* __restrict__ ks, const uint4* __restrict__ vs, uint4* __restrict__ kd,
            uint4* __restrict__ vd, int B, int count, int src_cap, int src_first, int dst_cap, int dst_first,
            int row_vecs) {
  const int lane = threadIdx.x & 31;
  const int rows_per_tensor = B * count;
  const int rows = 2 * rows_per_tensor;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const int t = r >= rows_per_tensor;
    const int e = r - (t ? rows_per_tensor : 0);
    const int b = e / count, i = e - b * count;
    const uint4* src = (t ? vs : ks) + ((int64_t)b * src_cap + src_first + i) * row_vecs;
    uint4* dst = (t ? vd : kd) + ((int64_t)b * dst_cap + dst_first + i) * row_vecs;
    for (int v0 = lane; v0 < row_vecs; v0 += 32 * kWriteUnroll) {
      uint4 val[kWriteUnroll];
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u)
        if (v0 + 32 * u < row_vecs) val[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u)
        if (v0 + 32 * u < row_vecs) dst[v0 + 32 * u] = val[u];
    }
  }
}

}  // namespace

cudaError_t kvc_launch_advance(kvc_cache* c, int row, int n, cudaStream_t s) {
  const kvc_config& g = c->cfg;
  return kvc_launch_pdl(k_advance, dim3(1), dim3(128), 0, s, c->meta, g.batch, row, n, g.layout, g.sink, g.window,
                        g.chunk, c->cap);
}

cudaError_t kvc_launch_reset(kvc_cache* c, int row, cudaStream_t s) {
  return kvc_launch_pdl(k_reset, dim3(1), dim3(128), 0, s, c->meta, c->cfg.batch, row);
}

cudaError_t kvc_launch_set_lengths(kvc_cache* c, const int32_t* kv_len, const int32_t* cu, cudaStream_t s) {
  return kvc_launch_pdl(k_set_lengths, dim3(1), dim3(128), 0, s, c->meta, c->cfg.batch, c->cap, kv_len, cu);
}

cudaError_t kvc_launch_set_lengths_block(int32_t* block, int B, int cap, const int32_t* kv_len, const int32_t* cu,
                                         cudaStream_t s) {
  return kvc_launch_pdl(k_set_lengths, dim3(1), dim3(128), 0, s, block, B, cap, kv_len, cu);
}

cudaError_t kvc_launch_write(kvc_cache* c, const void* k, const void* v, int n, const int32_t* slots,
                             cudaStream_t s) {
  const kvc_config& g = c->cfg;
  const int row_vecs = g.kv_heads * g.head_dim * c->eb / 16;
  const int64_t rows = 2LL * g.batch * n;
  int64_t blocks = (rows + kWriteThreads / 32 - 1) / (kWriteThreads / 32);
  const int64_t max_blocks = (int64_t)c->num_sms * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  return kvc_launch_pdl(k_write, dim3((unsigned)blocks), dim3(kWriteThreads), 0, s, (const uint4*)k, (const uint4*)v,
                        (uint4*)c->k, (uint4*)c->v, c->meta, c->lens, slots, g.batch, n, row_vecs, c->cap,
                        g.layout);
}

cudaError_t kvc_launch_write_rope(kvc_cache* c, const void* k, const void* v, int n, const int32_t* slots,
                                  const float* rope, int rope_positions, cudaStream_t s) {
  const kvc_config& g = c->cfg;
  const int row_vecs = g.kv_heads * g.head_dim * c->eb / 16;
  const int64_t tokens = (int64_t)g.batch * n;
  int64_t blocks = (tokens + kWriteThreads / 32 - 1) / (kWriteThreads / 32);
  const int64_t max_blocks = (int64_t)c->num_sms * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
#define KVC_WR(T)                                                                                               \
  kvc_launch_pdl(k_write_rope<T>, dim3((unsigned)blocks), dim3(kWriteThreads), 0, s, (const uint4*)k,          \
                 (const uint4*)v, (uint4*)c->k, (uint4*)c->v, c->meta, c->lens, slots, (const float2*)rope,     \
                 rope_positions, g.batch, n, row_vecs, c->cap, g.layout, g.chunk, g.head_dim)
  if (g.dtype == KVC_F32) return KVC_WR(float);
  if (g.dtype == KVC_F16) return KVC_WR(__half);
  return KVC_WR(__nv_bfloat16);
#undef KVC_WR
}

// One block moves ~100 GB/s: the single launch pays off for a decode step's bytes only.
bool kvc_append_fits(const kvc_cache* c, int n) {
  const int64_t bytes = 2LL * c->cfg.batch * n * c->cfg.kv_heads * c->cfg.head_dim * c->eb;
  return c->cfg.batch <= kAppendMaxRows && bytes <= (128 << 10);
}

cudaError_t kvc_launch_append(kvc_cache* c, const void* k, const void* v, int n, cudaStream_t s) {
  const kvc_config& g = c->cfg;
  const int row_vecs = g.kv_heads * g.head_dim * c->eb / 16;
  return kvc_launch_pdl(k_append, dim3(1), dim3(kWriteThreads), 0, s, (const uint4*)k, (const uint4*)v,
                        (uint4*)c->k, (uint4*)c->v, c->meta, g.batch, n, row_vecs, c->cap);
}

cudaError_t kvc_launch_roll(kvc_cache* c, void* scratch, cudaStream_t s) {
  const kvc_config& g = c->cfg;
  const int row_vecs = g.kv_heads * g.head_dim * c->eb / 16;
  const int count = g.window - g.sink - g.chunk;         // retained rolling tokens
  if (count <= 0) return cudaSuccess;
  const int64_t rows = 2LL * g.batch * count;
  int64_t blocks = (rows + kWriteThreads / 32 - 1) / (kWriteThreads / 32);
  const int64_t max_blocks = (int64_t)c->num_sms * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  uint4* sk = static_cast<uint4*>(scratch);
  uint4* sv = sk + (int64_t)g.batch * count * row_vecs;
  // clone: store rows [sink + chunk, window) -> scratch
  k_copy_rows<<<(unsigned)blocks, kWriteThreads, 0, s>>>((const uint4*)c->k, (const uint4*)c->v, sk, sv, g.batch,
                                                         count, c->cap, g.sink + g.chunk, count, 0, row_vecs);
  // copy back one chunk to the left: scratch -> store rows [sink, window - chunk)
  k_copy_rows<<<(unsigned)blocks, kWriteThreads, 0, s>>>(sk, sv, (uint4*)c->k, (uint4*)c->v, g.batch, count, count,
                                                         0, c->cap, g.sink, row_vecs);
  return cudaGetLastError();
}

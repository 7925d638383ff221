// Vocab-parallel embedding backward: the gradient of the masked shard lookup
// ("Vocab Parallelism" sec. 5.2.1) with respect to the tied weight, added to
// the LM head's gradient of the same parameter (sec. 5.2.2: embedding and LM
// head share one [V,H] weight, so its gradient is the sum of both layers').
//
// Shard t's lookup zeroes the output rows of ids outside its range, so those
// rows pass no gradient; every other token adds its upstream row dOut[n] into
// weight row id_n.  Summed over shards, each valid id's row receives exactly
// the upstream rows of the tokens carrying it:
//     dW[v,:] (+)= sum over n with id_n = v, in increasing n, of dOut[n,:]
// (fp32 accumulation; ids outside [0,V) contribute nothing).
//
// Deterministic, no atomics:
//   1. keys (id << 32 | n) for valid ids, all-ones for the rest and the
//      padding, sorted: blocks build and bitonic-sort 512-key chunks in shared
//      memory, then groups of up to 8 sorted runs merge in one pass each, every
//      key placing itself at its rank (binary searches in the other runs of its
//      group, held in shared memory for groups of up to 16384 keys; the keys
//      are distinct, the all-ones ones tie-broken by run).
//      The sorted order groups tokens by id, by n within.  This step needs only
//      the ids, so a caller can run it ahead (vp_embed_bwd_plan), off the
//      critical path, and the rest later (vp_embed_bwd_planned).
//   2. runs of kRun sorted positions: one thread per 16-byte column vector of
//      the row walks the run in order and sums; a segment (one id) that starts
//      and ends inside the run is added to dW at once, a segment cut by the
//      run's edge leaves its partial sum in a head or tail slot of the run.
//   3. the run that holds the start of a cut segment adds its tail, then the
//      head slots of the following runs up to the one where the segment ends,
//      in run order, and adds the total to dW.
// A row's sum is therefore taken in token order within runs of kRun sorted
// positions and over runs in order: the same bits on every call.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "vp_internal.h"

namespace vp {
namespace {

constexpr uint64_t kSentinel = ~0ull;
constexpr uint32_t kNoId = 0xffffffffu;
constexpr int kChunk = 512;           // keys sorted per block in shared memory
constexpr int kMergeWays = 8;         // sorted runs merged per pass
constexpr int kSortThreads = kChunk;   // one key per thread
constexpr int kRun = 32;              // sorted positions per run
constexpr int kRedThreads = 256;

__device__ __forceinline__ uint32_t key_id(uint64_t k) { return static_cast<uint32_t>(k >> 32); }

__device__ __forceinline__ uint64_t make_key(const int64_t* __restrict__ ids, int64_t N, int64_t V, int64_t i) {
  if (i >= N) return kSentinel;
  const int64_t id = ids[i];
  return (id >= 0 && id < V) ? (static_cast<uint64_t>(id) << 32) | static_cast<uint64_t>(i) : kSentinel;
}

// The keys of each chunk of len = min(kChunk, n_pad) positions, bitonic-sorted
// into ascending order (merge sizes 2..len), ready for the rank placement.
// One key per thread: compare-exchange partners less than a warp apart trade
// keys by shuffles, farther ones through shared memory.  A key's direction
// follows its index inside the chunk, so the last merge (k = len) leaves the
// chunk ascending.
__global__ void __launch_bounds__(kSortThreads) keys_chunk_sort(const int64_t* __restrict__ ids, int64_t N,
                                                                int64_t V, uint64_t* __restrict__ keys, int len) {
  __shared__ uint64_t s[kChunk];
  const int t = threadIdx.x;
  const int64_t gbase = static_cast<int64_t>(blockIdx.x) * len;
  uint64_t x = t < len ? make_key(ids, N, V, gbase + t) : kSentinel;
  for (int k = 2; k <= len; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      uint64_t y;
      if (j >= 32) {
        s[t] = x;
        __syncthreads();
        y = s[t ^ j];
        __syncthreads();
      } else {
        y = __shfl_xor_sync(0xffffffffu, x, j);
      }
      const bool asc = (t & k) == 0;
      const bool keep_min = ((t & j) == 0) == asc;
      x = keep_min ? (x < y ? x : y) : (x < y ? y : x);
    }
  }
  if (t < len) keys[gbase + t] = x;
}

// Merge each group of G consecutive sorted runs of L keys (G, L, n_pad powers
// of two, G * L dividing n_pad): a key's place in its group is its index in
// its own run plus, for every other run of the group, the keys there that
// precede it (an earlier run's equal keys first).  The G - 1 binary searches
// advance in lockstep, one independent load per run and round.
__global__ void rank_merge_kernel(const uint64_t* __restrict__ in, uint64_t* __restrict__ out, int64_t n_pad,
                                  int64_t L, int G) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_pad) return;
  const int64_t run = i / L;
  const int64_t first = run / G * G;
  const uint64_t key = in[i];
  int64_t lo[kMergeWays], hi[kMergeWays];
#pragma unroll
  for (int r = 0; r < kMergeWays; ++r) {
    lo[r] = 0;
    hi[r] = (r < G && first + r != run) ? L : 0;   // no search in the own run or past the group
  }
  for (int64_t span = L; span > 0; span >>= 1) {   // log2(L) + 1 rounds finish every search
#pragma unroll
    for (int r = 0; r < kMergeWays; ++r) {
      if (lo[r] < hi[r]) {
        const int64_t mid = (lo[r] + hi[r]) >> 1;
        const uint64_t x = in[(first + r) * L + mid];
        if (first + r < run ? x <= key : x < key)
          lo[r] = mid + 1;
        else
          hi[r] = mid;
      }
    }
  }
  int64_t pos = i - run * L;
#pragma unroll
  for (int r = 0; r < kMergeWays; ++r) pos += lo[r];
  out[first * L + pos] = key;
}

// The same placement with the group's runs first copied into shared memory
// (groups of up to kSmemMergeKeys keys): block b places keys [part * per,
// (part + 1) * per) of group b / parts, each by binary searches in the other
// runs held in shared memory.  Every block of a group copies the whole group.
constexpr int kSmemMergeKeys = 16384;   // 128 KB of keys
constexpr int kSmemMergeThreads = 512;
__global__ void __launch_bounds__(kSmemMergeThreads)
    rank_merge_smem_kernel(const uint64_t* __restrict__ in, uint64_t* __restrict__ out, int64_t L, int G, int parts) {
  extern __shared__ uint4 smem_keys[];
  const uint64_t* sg = reinterpret_cast<const uint64_t*>(smem_keys);
  const int64_t group = blockIdx.x / parts;
  const int part = static_cast<int>(blockIdx.x % parts);
  const int gsize = G * static_cast<int>(L);
  const uint4* src = reinterpret_cast<const uint4*>(in + group * gsize);
  const int nvec = gsize / 2;
  for (int base = threadIdx.x; base < nvec; base += 8 * blockDim.x) {   // 8 loads in flight per thread
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (base + u * static_cast<int>(blockDim.x) < nvec) v[u] = src[base + u * blockDim.x];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (base + u * static_cast<int>(blockDim.x) < nvec) smem_keys[base + u * blockDim.x] = v[u];
  }
  __syncthreads();
  const int per = gsize / parts, Li = static_cast<int>(L);
  for (int j = part * per + threadIdx.x; j < (part + 1) * per; j += blockDim.x) {
    const int run = j / Li;
    const uint64_t key = sg[j];
    int lo[kMergeWays], hi[kMergeWays];
#pragma unroll
    for (int r = 0; r < kMergeWays; ++r) {
      lo[r] = 0;
      hi[r] = (r < G && r != run) ? Li : 0;   // no search in the own run or past the group
    }
    for (int span = Li; span > 0; span >>= 1) {   // the searches advance in lockstep
#pragma unroll
      for (int r = 0; r < kMergeWays; ++r) {
        if (lo[r] < hi[r]) {
          const int mid = (lo[r] + hi[r]) >> 1;
          const uint64_t x = sg[r * Li + mid];
          if (r < run ? x <= key : x < key)
            lo[r] = mid + 1;
          else
            hi[r] = mid;
        }
      }
    }
    int pos = j - run * Li;
#pragma unroll
    for (int r = 0; r < kMergeWays; ++r) pos += lo[r];
    out[group * gsize + pos] = key;
  }
}

// 16 bytes of an upstream row as fp32 values: 8 bf16 or 4 f32.
template <int ESIZE>
struct Vec {
  static constexpr int kN = 16 / ESIZE;
  float v[kN];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int q = 0; q < kN; ++q) v[q] = 0.f;
  }
  __device__ __forceinline__ void add(const uint4& u) {
    if constexpr (ESIZE == 2) {
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[2 * q] += __uint_as_float(w[q] << 16);
        v[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
      }
    } else {
      v[0] += __uint_as_float(u.x);
      v[1] += __uint_as_float(u.y);
      v[2] += __uint_as_float(u.z);
      v[3] += __uint_as_float(u.w);
    }
  }
};

// dst[0..kN) += v (fp32, 16-byte aligned)
template <int ESIZE>
__device__ __forceinline__ void add_to(float* dst, const Vec<ESIZE>& a) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < Vec<ESIZE>::kN / 4; ++q) {
    float4 x = d[q];
    x.x += a.v[4 * q];
    x.y += a.v[4 * q + 1];
    x.z += a.v[4 * q + 2];
    x.w += a.v[4 * q + 3];
    d[q] = x;
  }
}
template <int ESIZE>
__device__ __forceinline__ void store_to(float* dst, const Vec<ESIZE>& a) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < Vec<ESIZE>::kN / 4; ++q)
    d[q] = make_float4(a.v[4 * q], a.v[4 * q + 1], a.v[4 * q + 2], a.v[4 * q + 3]);
}

__device__ __forceinline__ uint64_t key_at(const uint64_t* keys, int64_t n_pad, int64_t i) {
  return (i >= 0 && i < n_pad) ? keys[i] : kSentinel;
}

// Phase 2: grid (runs, column blocks); thread = one 16-byte vector column of H.
template <int ESIZE>
__global__ void __launch_bounds__(kRedThreads)
    embed_bwd_runs_kernel(const uint64_t* __restrict__ keys, int64_t n_pad, const uint4* __restrict__ dOut,
                          int64_t rowvec, float* __restrict__ dW, int64_t H, int64_t V, float* __restrict__ head,
                          float* __restrict__ tail) {
  __shared__ uint64_t sk[kRun + 2];
  const int64_t r = blockIdx.x;
  const int64_t p0 = r * kRun;
  for (int i = threadIdx.x; i < kRun + 2; i += blockDim.x) {
    const uint64_t k = key_at(keys, n_pad, p0 - 1 + i);
    sk[i] = key_id(k) < V ? k : kSentinel;   // an id outside [0, V) can only be a sentinel; never index dW with it
  }
  __syncthreads();
  const int64_t v = static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x;
  if (v >= rowvec || key_id(sk[1]) == kNoId) return;
  constexpr int kN = Vec<ESIZE>::kN;
  const int64_t col = v * kN;   // first fp32 column of this vector
  uint32_t cur = key_id(sk[1]);
  bool start_inside = key_id(sk[0]) != cur;
  Vec<ESIZE> acc;
  acc.zero();
  int i = 0;
#pragma unroll 1
  for (int i0 = 0; i0 < kRun; i0 += 8) {
    uint4 buf[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint64_t k = sk[1 + i0 + u];
      buf[u] = key_id(k) != kNoId ? __ldg(dOut + static_cast<int64_t>(k & 0xffffffffu) * rowvec + v)
                                  : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t id = key_id(sk[1 + i0 + u]);
      if (id == kNoId) break;
      if (id != cur) {   // the segment of `cur` ended inside this run
        if (start_inside)
          add_to<ESIZE>(dW + static_cast<int64_t>(cur) * H + col, acc);
        else
          store_to<ESIZE>(head + r * H + col, acc);
        cur = id;
        start_inside = true;
        acc.zero();
      }
      acc.add(buf[u]);
      i = i0 + u + 1;
    }
    if (i < i0 + 8) break;   // reached the sentinels
  }
  const bool ends_inside = key_id(sk[1 + i]) != cur;
  if (start_inside && ends_inside)
    add_to<ESIZE>(dW + static_cast<int64_t>(cur) * H + col, acc);
  else if (!start_inside)
    store_to<ESIZE>(head + r * H + col, acc);   // continued from an earlier run (it may run on past this one)
  else
    store_to<ESIZE>(tail + r * H + col, acc);   // starts here and continues into the next run
}

// Phase 3: the run holding the start of a segment cut at its end adds the
// segment's partials in run order.
template <int ESIZE>
__global__ void __launch_bounds__(kRedThreads)
    embed_bwd_cross_kernel(const uint64_t* __restrict__ keys, int64_t n_pad, int64_t rowvec,
                           float* __restrict__ dW, int64_t H, int64_t V, int64_t runs, const float* __restrict__ head,
                           const float* __restrict__ tail) {
  const int64_t r = blockIdx.x;
  const int64_t last = (r + 1) * kRun - 1;
  const uint32_t id = key_id(key_at(keys, n_pad, last));
  if (id >= V || key_id(key_at(keys, n_pad, last + 1)) != id) return;   // nothing continues past run r
  if (key_id(key_at(keys, n_pad, r * kRun - 1)) == id) return;              // the segment started earlier
  // The run where the segment ends (its head slot is the last part): the one
  // before the first later run whose first key has another id.  Warp 0 reads
  // the first keys of 32 runs at a time.
  __shared__ int64_t end_shared;
  if (threadIdx.x < 32) {
    int64_t e = -1;
    for (int64_t base = r + 1; e < 0 && base < runs; base += 32) {
      const int64_t q = base + threadIdx.x;
      const bool other = q >= runs || key_id(keys[q * kRun]) != id;
      const unsigned m = __ballot_sync(0xffffffffu, other);
      if (m) e = base + __ffs(m) - 2;
    }
    if (threadIdx.x == 0) end_shared = e < 0 ? runs - 1 : e;
  }
  __syncthreads();
  const int64_t end_run = end_shared;
  const int64_t v = static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x;
  if (v >= rowvec) return;
  constexpr int kN = Vec<ESIZE>::kN;
  const int64_t col = v * kN;
  // the tail of run r, then the head slots of runs r+1 .. end_run (8 runs'
  // 16-byte vectors in flight at a time), added in run order
  constexpr int kV4 = kN / 4;
  float4 s[kV4];
#pragma unroll
  for (int q = 0; q < kV4; ++q) s[q] = reinterpret_cast<const float4*>(tail + r * H + col)[q];
  for (int64_t r0 = r + 1; r0 <= end_run; r0 += 8) {
    float4 h[8][kV4];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int q = 0; q < kV4; ++q)
        h[u][q] = r0 + u <= end_run ? reinterpret_cast<const float4*>(head + (r0 + u) * H + col)[q]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (r0 + u <= end_run) {
#pragma unroll
        for (int q = 0; q < kV4; ++q) {
          s[q].x += h[u][q].x;
          s[q].y += h[u][q].y;
          s[q].z += h[u][q].z;
          s[q].w += h[u][q].w;
        }
      }
  }
  Vec<ESIZE> a;
#pragma unroll
  for (int q = 0; q < kV4; ++q) {
    a.v[4 * q] = s[q].x;
    a.v[4 * q + 1] = s[q].y;
    a.v[4 * q + 2] = s[q].z;
    a.v[4 * q + 3] = s[q].w;
  }
  add_to<ESIZE>(dW + static_cast<int64_t>(id) * H + col, a);
}

// The shared-memory merge's opt-in to kSmemMergeKeys keys of dynamic shared
// memory, made once per device.
cudaError_t allow_smem_merge() {
  static std::atomic<int> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(rank_merge_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemMergeKeys * sizeof(uint64_t)));
  if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
  return e;
}

int64_t pad_pow2(int64_t n) {
  int64_t p = 2;
  while (p < n) p <<= 1;
  return p;
}

}  // namespace

int embed_bwd_sort_kernels(int64_t N) {
  const int64_t n_pad = pad_pow2(N);
  int k = 1;   // keys + chunk sort
  for (int64_t L = n_pad < kChunk ? n_pad : kChunk; L < n_pad; L *= kMergeWays) ++k;   // merge passes
  return k;
}

size_t embed_bwd_workspace(int64_t N, int64_t H) {
  const int64_t runs = (N + kRun - 1) / kRun;
  return 2 * size_t(pad_pow2(N)) * sizeof(uint64_t) + 2 * size_t(runs) * H * sizeof(float);
}

// Step 1: the sorted keys, left in the workspace's first key buffer when the
// number of merge passes is even and in the second when it is odd
// (sorted_keys() finds them).
cudaError_t embed_bwd_sort(const int64_t* ids, int64_t N, int64_t V, void* workspace, cudaStream_t stream) {
  const int64_t n_pad = pad_pow2(N);
  uint64_t* keys = static_cast<uint64_t*>(workspace);   // two n_pad buffers, sorted in turn
  uint64_t* spare = keys + n_pad;
  const int len = static_cast<int>(n_pad < kChunk ? n_pad : kChunk);
  keys_chunk_sort<<<static_cast<unsigned>(n_pad / len), kSortThreads, 0, stream>>>(ids, N, V, keys, len);
  for (int64_t L = len; L < n_pad;) {
    const int G = static_cast<int>(n_pad / L < kMergeWays ? n_pad / L : kMergeWays);
    const int64_t gsize = G * L;
    if (gsize <= kSmemMergeKeys) {
      const size_t smem = size_t(gsize) * sizeof(uint64_t);
      if (smem > 48 * 1024) {
        const cudaError_t e = allow_smem_merge();
        if (e != cudaSuccess) return e;
      }
      const int parts = static_cast<int>(gsize / kChunk);   // kChunk keys placed per block
      rank_merge_smem_kernel<<<static_cast<unsigned>(n_pad / gsize * parts), kSmemMergeThreads, smem, stream>>>(
          keys, spare, L, G, parts);
    } else {
      rank_merge_kernel<<<static_cast<unsigned>((n_pad + 255) / 256), 256, 0, stream>>>(keys, spare, n_pad, L, G);
    }
    uint64_t* t = keys;
    keys = spare;
    spare = t;
    L *= G;
  }
  return cudaGetLastError();
}

namespace {
const uint64_t* sorted_keys(const void* workspace, int64_t N) {
  const int64_t n_pad = pad_pow2(N);
  const int passes = embed_bwd_sort_kernels(N) - 1;
  return static_cast<const uint64_t*>(workspace) + ((passes & 1) ? n_pad : 0);
}
}  // namespace

// Steps 2 and 3 on keys sorted by embed_bwd_sort into the same workspace.
cudaError_t embed_bwd_sums(const void* dOut, float* dW, int64_t N, int64_t H, int64_t V, int esize, bool accumulate,
                           void* workspace, cudaStream_t stream) {
  const int64_t n_pad = pad_pow2(N);
  const int64_t runs = (N + kRun - 1) / kRun;
  const uint64_t* keys = sorted_keys(workspace, N);
  float* head = reinterpret_cast<float*>(static_cast<uint64_t*>(workspace) + 2 * n_pad);
  float* tail = head + runs * H;
  cudaError_t e = cudaSuccess;
  if (!accumulate) e = cudaMemsetAsync(dW, 0, size_t(V) * H * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int64_t rowvec = H * esize / 16;
  const dim3 grid(static_cast<unsigned>(runs), static_cast<unsigned>((rowvec + kRedThreads - 1) / kRedThreads));
  const uint4* src = static_cast<const uint4*>(dOut);
  if (esize == 2) {
    embed_bwd_runs_kernel<2><<<grid, kRedThreads, 0, stream>>>(keys, n_pad, src, rowvec, dW, H, V, head, tail);
    embed_bwd_cross_kernel<2><<<grid, kRedThreads, 0, stream>>>(keys, n_pad, rowvec, dW, H, V, runs, head, tail);
  } else {
    embed_bwd_runs_kernel<4><<<grid, kRedThreads, 0, stream>>>(keys, n_pad, src, rowvec, dW, H, V, head, tail);
    embed_bwd_cross_kernel<4><<<grid, kRedThreads, 0, stream>>>(keys, n_pad, rowvec, dW, H, V, runs, head, tail);
  }
  return cudaGetLastError();
}

}  // namespace vp

// pkv_hash.cu -- chained prefix block hash ("ai-infra-7", "优化一：Prefix Cache",
// 工作原理：按块哈希):  h_0 = seed,  h_i = H(h_{i-1}, tokens of block i).
//
// H(p, blk) = fmix64(p XOR FNV1a64(bytes of blk)), the block's int32 tokens read
// as little-endian bytes.  FNV-1a is the Fowler/Noll/Vo hash (64-bit offset
// basis and prime); fmix64 is the SplitMix64 output mixer (Steele, Lea, Flood,
// OOPSLA 2014).  Splitting H this way lets every block digest be computed in
// parallel; only the cheap mixing chain is sequential, as the definition
// requires.  One CTA per sequence: threads digest blocks into shared memory, one
// thread runs the chain over each chunk of digests.
#include "pkv_internal.cuh"

namespace pkv {

constexpr int kHashChunk = 2048;   // digests staged in shared memory per pass (16 KB)

__device__ __forceinline__ uint64_t fnv1a64_tokens(const int32_t* tok, int n) {
    uint64_t h = 14695981039346656037ull;   // FNV-64 offset basis
    for (int j = 0; j < n; ++j) {
        const uint32_t w = (uint32_t)tok[j];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            h ^= (uint64_t)((w >> (8 * b)) & 0xFFu);
            h *= 1099511628211ull;          // FNV-64 prime
        }
    }
    return h;
}

__device__ __forceinline__ uint64_t fmix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

__global__ void __launch_bounds__(256)
    pkv_prefix_hash_kernel(const int32_t* __restrict__ tokens, const int64_t* __restrict__ offsets,
                           int B, uint64_t seed, uint64_t* __restrict__ hashes,
                           const int64_t* __restrict__ hash_offsets) {
    __shared__ uint64_t dig[kHashChunk];
    const int s = blockIdx.x;
    const int64_t begin = offsets[s];
    const int64_t len = offsets[s + 1] - begin;
    const int64_t nb = len / B;
    uint64_t* out = hashes + hash_offsets[s];
    uint64_t h = seed;
    for (int64_t c0 = 0; c0 < nb; c0 += kHashChunk) {
        const int n = (int)min((int64_t)kHashChunk, nb - c0);
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            dig[i] = fnv1a64_tokens(tokens + begin + (c0 + i) * B, B);
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int i = 0; i < n; ++i) {
                h = fmix64(h ^ dig[i]);
                out[c0 + i] = h;
            }
        }
        __syncthreads();
    }
}

cudaError_t prefix_hash_launch(const int32_t* tokens, const int64_t* offsets, int num_seqs, int B,
                               uint64_t seed, uint64_t* hashes, const int64_t* hash_offsets,
                               cudaStream_t st) {
    if (num_seqs == 0) return cudaSuccess;
    pkv_prefix_hash_kernel<<<num_seqs, 256, 0, st>>>(tokens, offsets, B, seed, hashes,
                                                     hash_offsets);
    return cudaGetLastError();
}

}  // namespace pkv

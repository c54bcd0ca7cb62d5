// pkv_hash.cu -- chained prefix block hash ("ai-infra-7", "优化一：Prefix Cache",
// 工作原理：按块哈希):  h_0 = seed,  h_i = H(h_{i-1}, tokens of block i).
//
// H(p, blk) = fmix64(p XOR FNV1a64(bytes of blk)), the block's int32 tokens read
// as little-endian bytes.  FNV-1a is the Fowler/Noll/Vo hash (64-bit offset
// basis and prime); fmix64 is the SplitMix64 output mixer (Steele, Lea, Flood,
// OOPSLA 2014).  Splitting H this way lets every block digest be computed in
// parallel; only the cheap mixing chain is sequential, as the definition
// requires.  One CTA per sequence.  Digests are staged in shared memory chunk by
// chunk, double-buffered: warps 1-7 digest chunk c + 1 while lane 0 of warp 0 runs
// the chain over chunk c, so a long sequence costs about its chain (tens of cycles
// per block) rather than chain plus digests.
#include "pkv_internal.cuh"

namespace pkv {

constexpr int kHashChunk = 2048;    // digests per shared-memory buffer (16 KB)
constexpr int kHashThreads = 256;

__device__ __forceinline__ uint64_t fnv1a64_word(uint64_t h, uint32_t w) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        h ^= (uint64_t)((w >> (8 * b)) & 0xFFu);
        h *= 1099511628211ull;              // FNV-64 prime
    }
    return h;
}

// FNV-1a 64 over the little-endian bytes of n int32 tokens; the loads of each group
// of eight tokens are issued together before they are hashed
__device__ __forceinline__ uint64_t fnv1a64_tokens(const int32_t* tok, int n) {
    uint64_t h = 14695981039346656037ull;   // FNV-64 offset basis
    int j = 0;
    for (; j + 8 <= n; j += 8) {
        uint32_t w[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) w[t] = (uint32_t)__ldg(tok + j + t);
#pragma unroll
        for (int t = 0; t < 8; ++t) h = fnv1a64_word(h, w[t]);
    }
    for (; j < n; ++j) h = fnv1a64_word(h, (uint32_t)__ldg(tok + j));
    return h;
}

__device__ __forceinline__ uint64_t fmix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// Full chain (prev_hashes == nullptr): every full block of the sequence, from h_0 =
// seed.  Resumed chain: the first max(first_blocks[s], 0) full blocks were hashed
// before and prev_hashes[s] is the last of them (h_k), so only the blocks after them
// are digested and chained.  Either way at most hash_offsets[s+1] - hash_offsets[s]
// hashes are written.
__global__ void __launch_bounds__(kHashThreads)
    pkv_prefix_hash_kernel(const int32_t* __restrict__ tokens, const int64_t* __restrict__ offsets,
                           int B, uint64_t seed, const uint64_t* __restrict__ prev_hashes,
                           const int64_t* __restrict__ first_blocks,
                           uint64_t* __restrict__ hashes,
                           const int64_t* __restrict__ hash_offsets) {
    __shared__ uint64_t dig[2][kHashChunk];
    const int s = blockIdx.x;
    const int64_t full = (offsets[s + 1] - offsets[s]) / B;
    int64_t k = 0;
    uint64_t h0 = seed;
    if (prev_hashes) {
        k = first_blocks[s];
        k = k < 0 ? 0 : (k > full ? full : k);
        h0 = prev_hashes[s];
    }
    const int64_t room = hash_offsets[s + 1] - hash_offsets[s];
    int64_t nb = full - k;                      // blocks to hash, from block k (0-based)
    if (nb > room) nb = room;
    if (nb < 0) nb = 0;
    const int64_t begin = offsets[s] + k * B;
    const int nchunks = (int)((nb + kHashChunk - 1) / kHashChunk);
    uint64_t* out = hashes + hash_offsets[s];
    // digests of chunk c into buffer c & 1, by threads [t0, kHashThreads)
    auto digest = [&](int c, int t0) {
        const int64_t c0 = (int64_t)c * kHashChunk;
        const int n = (int)min((int64_t)kHashChunk, nb - c0);
        for (int i = (int)threadIdx.x - t0; i < n; i += kHashThreads - t0)
            dig[c & 1][i] = fnv1a64_tokens(tokens + begin + (c0 + i) * B, B);
    };
    if (nchunks > 0) digest(0, 0);
    __syncthreads();
    uint64_t h = h0;
    for (int c = 0; c < nchunks; ++c) {
        if (threadIdx.x < 32) {
            if (threadIdx.x == 0) {
                const int64_t c0 = (int64_t)c * kHashChunk;
                const int n = (int)min((int64_t)kHashChunk, nb - c0);
                const uint64_t* d = dig[c & 1];
                uint64_t* o = out + c0;
                // eight digests read ahead of the chain, so only fmix64's own latency
                // is sequential
                int i = 0;
                for (; i + 8 <= n; i += 8) {
                    uint64_t w[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) w[t] = d[i + t];
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        h = fmix64(h ^ w[t]);
                        o[i + t] = h;
                    }
                }
                for (; i < n; ++i) {
                    h = fmix64(h ^ d[i]);
                    o[i] = h;
                }
            }
        } else if (c + 1 < nchunks) {
            digest(c + 1, 32);
        }
        __syncthreads();
    }
}

cudaError_t prefix_hash_launch(const int32_t* tokens, const int64_t* offsets, int num_seqs, int B,
                               uint64_t seed, const uint64_t* prev_hashes,
                               const int64_t* first_blocks, uint64_t* hashes,
                               const int64_t* hash_offsets, cudaStream_t st) {
    if (num_seqs == 0) return cudaSuccess;
    pkv_prefix_hash_kernel<<<num_seqs, kHashThreads, 0, st>>>(tokens, offsets, B, seed, prev_hashes,
                                                              first_blocks, hashes, hash_offsets);
    return cudaGetLastError();
}

}  // namespace pkv

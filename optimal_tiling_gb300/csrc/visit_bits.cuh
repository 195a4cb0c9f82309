// The set of key (or query) blocks a CTA visits under a block mask, held as a
// bit set in shared memory.  Built once per CTA by all its warps together (one
// mask entry per lane, one __ballot_sync per 32 blocks), then walked by every
// role with find-first-set.  Reading the mask entry by entry in each thread
// instead costs one dependent global load per block before any work starts,
// which dominates a CTA that visits only a few blocks of a long mask row.
#pragma once

#include <stdint.h>

namespace attn {

struct VisitBits {
    const uint32_t *words;  // shared memory, bit b of word w = block 32 w + b
    int nwords;

    // Number of visited blocks (every thread may call it; reads shared memory only).
    __device__ __forceinline__ int count() const {
        int n = 0;
        for (int w = 0; w < nwords; ++w) n += __popc(words[w]);
        return n;
    }
    // First visited block after j (j = -1 for the first).  Callers ask only while one remains.
    __device__ __forceinline__ int next(int j) const {
        int w = (j + 1) >> 5;
        uint32_t bits = words[w] & (0xFFFFFFFFu << ((j + 1) & 31));
        while (bits == 0) bits = words[++w];
        return (w << 5) + __ffs(bits) - 1;
    }
};

// All threads of the CTA call this (it ends with no barrier: the caller's next
// __syncthreads publishes the words).  visited(b) must be valid for b < nbits.
template <class Pred>
__device__ __forceinline__ void build_visit_bits(uint32_t *words, int nbits, Pred visited) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int nwords = (nbits + 31) >> 5;
    for (int w = warp; w < nwords; w += nwarps) {
        const int b = (w << 5) + lane;
        const uint32_t bits = __ballot_sync(0xFFFFFFFFu, b < nbits && visited(b));
        if (lane == 0) words[w] = bits;
    }
}

}  // namespace attn

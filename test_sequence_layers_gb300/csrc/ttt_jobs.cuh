// ttt_jobs.cuh -- the order in which a (batch, head) chain's tokens are processed.
//
// A mini-batch of b tokens (the last one may be shorter) is cut into chunks of at
// most 16 tokens, the row count of one tensor-core tile.  Every role of a CTA
// (producer, score warp, chain warps) walks the same job list, so a job index
// names one pipeline stage use.
//
//   causal, or a mini-batch of a single chunk:
//       one kBoth job per chunk (update the weights and produce the chunk's outputs)
//   non-causal mini-batch of several chunks (queries read the block-end weights):
//       kUpd jobs for every chunk, then kOut jobs for every chunk.
#pragma once

namespace ttt {

enum JobKind : int { kBoth = 0, kUpd = 1, kOut = 2 };

struct Job {
    int t0;          // first token of the chunk
    int c;           // tokens in the chunk (1..16)
    int kind;        // JobKind
    int first;       // first chunk of its pass over the mini-batch
    int last_of_mb;  // last job of the mini-batch
    int last_upd;    // last job of the mini-batch that updates the weights
};

struct JobIter {
    int T, b, causal;
    int n0, L, nch, njobs, j;

    __device__ __forceinline__ JobIter(int T_, int b_, int causal_)
        : T(T_), b(b_), causal(causal_), n0(0), L(0), nch(0), njobs(0), j(0)
    {
        if (T > 0) setup();
    }
    __device__ __forceinline__ void setup()
    {
        L = min(b, T - n0);
        nch = (L + 15) >> 4;
        njobs = (causal || nch == 1) ? nch : 2 * nch;
        j = 0;
    }
    __device__ __forceinline__ bool valid() const { return n0 < T; }
    __device__ __forceinline__ Job get() const
    {
        Job o;
        const bool split = !(causal || nch == 1);
        const int ch = (split && j >= nch) ? j - nch : j;
        o.t0 = n0 + 16 * ch;
        o.c = min(16, L - 16 * ch);
        o.kind = !split ? kBoth : (j < nch ? kUpd : kOut);
        o.first = (ch == 0);
        o.last_of_mb = (j == njobs - 1);
        o.last_upd = split ? (j == nch - 1) : o.last_of_mb;
        return o;
    }
    __device__ __forceinline__ void next()
    {
        if (++j == njobs) {
            n0 += b;  // b <= T (clamped by the host), so this cannot overflow
            if (n0 < T) setup();
        }
    }
};

}  // namespace ttt

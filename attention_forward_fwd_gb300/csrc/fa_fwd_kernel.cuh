// fa_fwd_kernel.cuh -- FlashAttention-2 forward kernel for sm_103a.
//
// What it computes (page "CuTe 详解：以 FlashAttention-2 拆解 Layout、TiledCopy
// 与 TiledMMA"): per query tile, S = Q K^T, P = softmax(S), O = P V (section
// 先看全局), carried across key tiles with the running max m_i, running sum
// l_i and unnormalised output o~_i of section 教学配置, updated with
// alpha = exp(m_old - m_new) as in section 沿 C fragment 做 Online Softmax,
// and normalised O = o~ / l only after the last key tile.  The max is taken
// on the raw scores and the positive scale folded in afterwards (same
// section, last paragraph), as exp2 with scale*log2(e) folded into one FMA.
//
// How it maps onto one GB300 SM (one CTA per SM; RS softmax threads per
// query row, RS = 1 or 2, 128*(2*RS+1) threads):
//   warps [0, 4RS)     softmax for query tile 0 (rows q0 .. q0+127): each row
//                      (a TMEM lane) is handled by RS threads, one per 128/RS
//                      score columns.  They also rescale O in TMEM when the
//                      row max moves and run the epilogue of the tile.
//   warps [4RS, 8RS)   the same for query tile 1 (rows q0+128 .. q0+255).
//   warp  8RS          MMA issuer (the whole warp runs the loop, one
//                      elected lane issues): S_t = Q_t K_j^T and
//                      O_t += P_t V_j with tcgen05.mma, accumulators in TMEM;
//                      allocates TMEM.  With separate P (below) it issues for
//                      query tile 0 only and
//   warp  8RS+2        issues for query tile 1.
//   warp  8RS+1        TMA producer (one thread): Q tiles once, then K_j / V_j
//                      tiles through an NS-slot ring paced by full/empty
//                      mbarriers.
//   warp  8RS+3        idle (completes the control warpgroup).
// TMEM (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256),
// O_0 [256,256+D), O_1 [256+D,256+2D).  P_t (16-bit, packed in pairs) is
// written over the first 64 columns of S_t and read from there as the A
// operand of the second product; V stays [key][d] in shared memory and is
// read as an MN-major B operand (the transpose is only a view, section
// V 的转置只发生在视图里).
//
// Every wait is bounded in time.  A wait that runs out sets a shared abort
// flag and the device status word; every role then stops issuing work, waits
// (again bounded) for what it already has in flight, and the CTA frees its
// TMEM and exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBM = 128;              // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;              // keys per tile
constexpr int kQTiles = 2;            // query tiles per CTA
// Warp roles for RS softmax threads per query row (RS = 1: one thread per
// row; RS = 2: each row split into two column halves).  Warps [0, 8*RS) run
// the softmax, the last warpgroup holds the MMA issuers and the TMA producer.
// Register budget: the kernel launches with kLaunchRegs per thread (checked
// against ptxas by the build); the softmax warpgroups then take kSoftmaxRegs
// and the control warpgroup gives back down to kControlRegs, within the
// launch total.
template <int RS>
struct WarpLayout;
template <>
struct WarpLayout<1> {
    static constexpr int kSoftmaxWarps = 8;
    static constexpr uint32_t kLaunchRegs = 168;
    static constexpr uint32_t kSoftmaxRegs = 224;
    static constexpr uint32_t kControlRegs = 56;
};
template <>
struct WarpLayout<2> {
    static constexpr int kSoftmaxWarps = 16;
    static constexpr uint32_t kLaunchRegs = 96;
    static constexpr uint32_t kSoftmaxRegs = 104;
    static constexpr uint32_t kControlRegs = 64;
};
template <int RS>
struct Roles : WarpLayout<RS> {
    using B = WarpLayout<RS>;
    static constexpr int kThreads = 32 * B::kSoftmaxWarps + 128;
    static constexpr int kMmaWarp = B::kSoftmaxWarps;       // MMA issuer, tile 0; TMEM alloc
    static constexpr int kLoadWarp = B::kSoftmaxWarps + 1;  // TMA producer
    static constexpr int kMmaWarp1 = B::kSoftmaxWarps + 2;  // MMA issuer, tile 1
    static constexpr int kTileThreads = 128 * RS;           // softmax threads per query tile
    static_assert(32u * B::kSoftmaxWarps * B::kSoftmaxRegs + 128u * B::kControlRegs <=
                      kThreads * B::kLaunchRegs,
                  "register split exceeds the launch budget");
};
constexpr uint32_t kTmemCols = 512;
constexpr float kTauLog2 = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr float kMaxTileSum = 256.0f;  // 2^kTauLog2: a tile's row sum that keeps the reference
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s per wait

constexpr int kStatusTimeout = 4;
constexpr int kStatusBadSeqlens = 5;   // a sequence offset was out of range (sequence skipped)

constexpr int kStatusDeviceCheck = 6;   // a device-side invariant check failed (FA_DEBUG builds)

// Device status word: 0, or the status of the first wait that ran out.
__device__ int g_fa_device_status;

// Builds with FA_DEBUG = 1 check invariants on the device (work-item bounds,
// the tensor-memory allocation, the roles' tile counts, row sums); a failed
// check records kStatusDeviceCheck in the status word -- the kernel does not
// trap -- and the results are those of the build without the checks.
#ifndef FA_DEBUG
#define FA_DEBUG 0
#endif
__device__ __forceinline__ void debug_check(bool cond) {
    if constexpr (FA_DEBUG != 0) {
        if (!cond) atomicCAS(&g_fa_device_status, 0, kStatusDeviceCheck);
    }
}

// query blocks per head, and work items per head, beyond which the keys are
// never split
constexpr int kMaxSplitBlocks = 128;
constexpr int kMaxSplitItems = 256;

struct FwdParams {
    int B, H, S;
    // The caller's head dimension (a multiple of 8, at most the kernel's D).
    // The tensor maps cover only these columns: TMA reads the others as
    // zeros and drops them on the O stores, so S and O are exact; the direct
    // stores below use it for the row stride and skip the columns past it.
    int d_head;
    int causal;
    int kv_group;       // query heads per K/V head (K, V have H / kv_group heads)
    // Local attention: key j is kept for query i iff i - win_left <= j <= i +
    // win_right (-1: no bound on that side; the causal mask caps the right
    // bound at 0).  Windowed calls are not split over keys.
    int win_left, win_right;
    // Variable-length batch (cu_seqlens != nullptr): Q, K, V, O are packed
    // [total, heads, D], sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1
    // (at most S rows), LSE is [H, total].  Work items of query blocks past a
    // sequence's end are empty and skipped.
    const int* cu_seqlens;
    int total;
    void* o_ptr;        // O, for the row-by-row stores of a sequence's last tile
    // Test support (fa_selftest_timeout): 1 = the first item's Q is never
    // loaded, so the waits on it run out and the kernel must end in the
    // timeout status instead of hanging.  0 in every other call.
    int drop_first_q;
    // Attention dropout (dropout variant only): each Philox4x32-10 word holds
    // two 16-bit draws (low half first), so the block with counter (j / 8, i,
    // h, b) and the 64-bit seed as key serves keys 8 (j / 8) .. + 7; P(i, j)
    // of head (b, h) is kept iff draw j % 8 is >= floor(p * 2^16), held here
    // shifted up by 16 bits.  Kept values are scaled by drop_inv_keep =
    // 1 / (1 - p); the row sum and LSE are those of the undropped softmax.
    uint32_t drop_seed_lo, drop_seed_hi;
    uint32_t drop_threshold;
    float drop_inv_keep;
    // Work items: the (query block, split) pairs of every head, numbered
    // w = y * (B*H) + b*H + h with y the block's visit index (heaviest first
    // when causal).  Each CTA runs items blockIdx.x, 2G-1-blockIdx.x,
    // 2G+blockIdx.x, ... (G = gridDim.x, every other round reversed), so a
    // grid of one CTA per SM keeps its set-up across items and the rounds of
    // heavy and light blocks even out.
    int items;
    float scale_log2;   // scale * log2(e)
    float* lse;         // [B, H, S] fp32 or nullptr
    // Split over keys (kv_chunk = 0: off).  In split mode the work items of a
    // head are (query block, split) pairs in the order of split_item; query
    // block qb with T key tiles and n splits gives split s the key tiles
    // [s*c, min(T, (s+1)*c)), c = ceil(T / n).  A block with more than one
    // split writes partial results (see partial_slot) that fa_combine_kernel
    // merges.
    int nqb;            // query blocks of kQTiles*kBM rows per head
    int kv_chunk;       // nonzero: split mode
    int max_splits;     // splits of the most split query block
    float* ws_o;        // partial o~ tiles (fp32)
    float* ws_ml;       // partial (m * scale * log2e, l) per row
    // split mode: item y of a head is split (split_item[y] >> 8) & 0xfff of
    // query block split_item[y] & 0xff, which has split_item[y] >> 20 splits.
    // One table entry per item: the decode takes one load, not a search (a
    // chain of dependent parameter loads is slow right after launch).
    uint32_t split_item[kMaxSplitItems];
    uint8_t block_splits[kMaxSplitBlocks];   // splits of each query block
};

// Workspace of the split-over-keys path.  One partial slot per (b*H + h,
// query tile qt of 128 rows, split s):
//   slot = ((bh * ntq) + qt) * max_splits + s,   ntq = ceil(S / 128)
//   ws_o  + slot * 128 * D  : o~ rows, fp32, as [D/4][128] float4 (column
//                             chunk major, so a warp's stores are contiguous)
//   ws_ml + slot * 256      : [0,128) m in log2 units, [128,256) l
// A tile that saw no key in a split records l = 0 (and m = -inf).
__host__ __device__ inline size_t partial_slot(int bh, int ntq, int qt, int max_splits, int s) {
    return (static_cast<size_t>(bh) * ntq + qt) * max_splits + s;
}

// Key tiles (of kBN) that a query tile starting at row r0 visits: all tiles
// holding a key < S, or, when causal, up to the tile holding its last row.
__host__ __device__ inline int key_tiles_for(int r0, int S, bool causal) {
    const int nkv_all = (S + kBN - 1) / kBN;
    if (r0 >= S) return 0;
    return causal ? min(nkv_all, (r0 + kBM - 1) / kBN + 1) : nkv_all;
}

// Key tiles of a query block (the longest of its kQTiles query tiles).
__host__ __device__ inline int key_tiles_for_block(int qb, int S, bool causal) {
    int n = 0;
    for (int t = 0; t < kQTiles; ++t) n = max(n, key_tiles_for(qb * kQTiles * kBM + t * kBM, S, causal));
    return n;
}

// P_t in TMEM columns of its own (when 2*kBN + 2*D + kQTiles*kBN/2 fit in
// 512, i.e. D = 64), else written over S_t.
__host__ __device__ constexpr bool separate_p(int D) {
    return (2 * kBN + 2 * D + kQTiles * (kBN / 2)) <= static_cast<int>(kTmemCols);
}

template <int NS, int RS>
struct Barriers {
    uint64_t q_full;
    uint64_t q_empty;   // the Q buffer may be loaded with the next item's Q
    uint64_t kv_full[NS];
    uint64_t kv_empty[NS];
    uint64_t s_full[kQTiles];
    uint64_t s_free[kQTiles];   // S_t read into registers (separate-P schedule)
    uint64_t p_full[kQTiles];
    uint64_t p_half[kQTiles];   // separate P: the first half of P_t (keys 0..63) is stored
    uint64_t o_done[kQTiles];
    uint64_t drain[kQTiles];
    uint32_t tmem_base;
    int abort;
    // FA_DEBUG: tiles each role saw (producer ring, each issuer's ring, S per
    // query tile as issued and as read by the softmax)
    int dbg[7];
    // the RS threads of a row swap partial row maxima (double-buffered over
    // key tiles) and, at the end of an item, partial row sums (double-buffered
    // over items)
    float row_max[2][kQTiles][RS][kBM];
    float row_sum[2][kQTiles][RS][kBM];
};

// Shared memory: Q tiles, the K / V ring and, where there is room (D = 64),
// a buffer of its own for staging the O tiles of the TMA-store epilogue, so
// that the next item's Q can be loaded while the O of this one is stored.
// Where there is none (D = 128) the softmax threads store their O rows to
// global memory themselves (kDirectO), so that the Q buffer is free once the
// item's last S = Q K^T has run; the other choice (kStageInQ) stages O in
// the Q buffer it replaces, and the next Q waits for that store.
#ifndef FA_DIRECT_O_D128
#define FA_DIRECT_O_D128 1
#endif
template <int D, int NS, int RS>
struct SmemLayout {
    static constexpr int kQBytes = kBM * D * 2;
    static constexpr int kKVBytes = kBN * D * 2;
    static constexpr bool kDirectO = !separate_p(D) && FA_DIRECT_O_D128;
    static constexpr bool kStageInQ = !separate_p(D) && !kDirectO;
    static constexpr bool kOwnStage = !kDirectO && !kStageInQ;
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kQTiles * kQBytes;
    static constexpr int kOffStage = kOwnStage ? kOffKV + NS * kKVBytes : kOffQ;
    static constexpr int kOffBar = kOffKV + NS * kKVBytes + (kOwnStage ? kQTiles * kQBytes : 0);
    static constexpr int kBytes = kOffBar + static_cast<int>(sizeof(Barriers<NS, RS>));
    static constexpr int kAlloc = kBytes + 1024;   // slack to align the base to 1024
    static_assert(kAlloc <= 232448, "shared memory beyond the 227 KiB a CTA may use");
};

// One work item: a query block of kQTiles*kBM rows of head (b, h) and the
// key tiles [jb, jb + nkv_t) that query tile t visits in this item's split.
struct WorkItem {
    int b, h, bh;
    int hkv;            // the K/V head of query head h
    int S;              // rows of this item's sequence
    int base;           // first row of the sequence in the (packed) tensors
    int tb;             // batch coordinate of the tensor maps (0 when packed)
    bool bad;           // its sequence offsets were out of range
    int q0;             // first query row of the block
    int jb;             // first key tile of the split
    // query tile t uses key tiles [s_t, nkv_t) of the item's range (counted
    // from jb); s_t > 0 only with a left window bound
    int s0, s1;
    int nkv0, nkv1;
    int nkv;            // max(nkv0, nkv1): the item's key tiles through the ring
    int split;          // split index within the block
    bool partial;       // the block is split: write partial results
};

// Kernel variants: the plain batched call, packed variable-length batches,
// local (sliding-window) attention and attention dropout; each compiles only
// its own extras.
enum Feature : int { kPlain = 0, kPacked = 1, kLocal = 2, kDropout = 3 };

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): ten rounds of two 32x32 -> 64-bit products,
// the key bumped by the Weyl constants between rounds.
// N blocks with counters (g0 + n, c1, c2, c3) side by side, so that the
// compiler can interleave their rounds (each round is a chain of two wide
// multiplies and two XORs; one block alone leaves the SM waiting on it).
// Word k of block n goes to w[4 n + k].
template <int N>
__device__ __forceinline__ void philox4x32_10(uint32_t g0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              uint32_t k0, uint32_t k1, uint32_t (&w)[4 * N]) {
    constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
    constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
    for (int n = 0; n < N; ++n) {
        w[4 * n + 0] = g0 + n;
        w[4 * n + 1] = c1;
        w[4 * n + 2] = c2;
        w[4 * n + 3] = c3;
    }
#pragma unroll
    for (int r = 0; r < 10; ++r) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
            uint32_t* c = w + 4 * n;
            const uint32_t hi0 = __umulhi(kM0, c[0]), lo0 = kM0 * c[0];
            const uint32_t hi1 = __umulhi(kM1, c[2]), lo1 = kM1 * c[2];
            const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
            c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
        }
        k0 += kW0; k1 += kW1;
    }
}

template <int FEAT>
__device__ __forceinline__ WorkItem decode_item(const FwdParams& p, int w) {
    WorkItem it;
    const int bhn = p.B * p.H;
    const int y = w / bhn;
    it.bh = w - y * bhn;
    it.b = it.bh / p.H;
    it.h = it.bh - it.b * p.H;
    it.hkv = it.h / p.kv_group;
    it.S = p.S;
    it.base = 0;
    it.tb = it.b;
    it.bad = false;
    if constexpr (FEAT == kPacked) {
        const int a = p.cu_seqlens[it.b];
        const int e = p.cu_seqlens[it.b + 1];
        // offsets outside [0, total], decreasing, or a sequence longer than S:
        // nothing of it is read or written
        it.bad = !(a >= 0 && e >= a && e <= p.total && e - a <= p.S);
        it.S = it.bad ? 0 : e - a;
        it.base = it.bad ? 0 : a;
        it.tb = 0;
    }
    const bool causal = p.causal != 0;
    int qb, je, nsplit;
    if (p.kv_chunk <= 0) {
        qb = causal ? (p.nqb - 1 - y) : y;   // causal: heaviest query blocks first
        it.jb = 0;
        je = 0x7fffffff;
        nsplit = 1;
        it.split = 0;
    } else {
        const uint32_t e = p.split_item[y];
        qb = static_cast<int>(e & 0xffu);
        nsplit = static_cast<int>(e >> 20);
        it.split = static_cast<int>((e >> 8) & 0xfffu);
        const int chunk = (key_tiles_for_block(qb, it.S, causal) + nsplit - 1) / nsplit;
        it.jb = it.split * chunk;
        je = it.jb + chunk;
    }
    it.q0 = qb * (kQTiles * kBM);
    it.nkv0 = max(0, min(je, key_tiles_for(it.q0, it.S, causal)) - it.jb);
    it.nkv1 = max(0, min(je, key_tiles_for(it.q0 + kBM, it.S, causal)) - it.jb);
    it.s0 = it.s1 = 0;
    if constexpr (FEAT == kLocal) {
        // key tiles [lo_t, hi_t) that query tile t's rows reach (jb is 0 here)
        int lo[kQTiles], hi[kQTiles];
        for (int t = 0; t < kQTiles; ++t) {
            const int r0 = it.q0 + t * kBM;
            const int e = t == 0 ? it.nkv0 : it.nkv1;
            lo[t] = p.win_left < 0 ? 0 : max(0, r0 - p.win_left) / kBN;
            hi[t] = p.win_right < 0 ? e : min(e, (r0 + kBM - 1 + p.win_right) / kBN + 1);
            if (hi[t] <= lo[t]) lo[t] = hi[t] = 0;   // no key for this tile
        }
        const int first = hi[0] > 0 ? lo[0] : lo[1];
        it.jb = first;
        it.s0 = hi[0] > 0 ? lo[0] - first : 0;
        it.nkv0 = hi[0] > 0 ? hi[0] - first : 0;
        it.s1 = hi[1] > 0 ? lo[1] - first : 0;
        it.nkv1 = hi[1] > 0 ? hi[1] - first : 0;
    }
    it.nkv = max(it.nkv0, it.nkv1);
    it.partial = nsplit > 1;
    if constexpr (FA_DEBUG != 0) {
        // key tiles [jb, jb + nkv) inside the sequence, each query tile's
        // range inside the item's, and the split fields in range
        const int tiles = (it.S + kBN - 1) / kBN;
        debug_check(it.jb >= 0 && it.s0 >= 0 && it.s1 >= 0 && it.s0 <= it.nkv0 && it.s1 <= it.nkv1 &&
                    (it.nkv == 0 || (it.jb + it.nkv <= tiles && it.q0 < it.S)));
        if (p.kv_chunk > 0) debug_check(qb < p.nqb && nsplit >= 1 && it.split < nsplit);
    }
    return it;
}

// Item index of this CTA's k-th work item, or -1 past its last one.
__device__ __forceinline__ int cta_item(int k, int items) {
    const long long G = gridDim.x;
    const long long c = blockIdx.x;
    const long long w = k * G + ((k & 1) ? (G - 1 - c) : c);
    return w < items ? static_cast<int>(w) : -1;
}

// Bounded wait on the phase of `bar` with parity `parity`.  Returns false
// (and sets the abort flag) if the wait ran out of time, or false at once if
// another role already aborted and `honour_abort` is set.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           bool honour_abort = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((n & 31u) == 0) {
            if (honour_abort && *abort_flag) return false;
            if (ptx::globaltimer() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicCAS(&g_fa_device_status, 0, kStatusTimeout);
                return false;
            }
        }
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Dropout draws for the keys col0 .. col0 + 8 N - 1 (col0 % 8 == 0) of query
// row `row`: N Philox blocks, counters (col0 / 8 + n, row, h, b).  Word k of
// block n holds the draws of keys col0 + 8 n + 2 k (low half) and + 1 (high).
template <int N>
__device__ __forceinline__ void drop_words(const FwdParams& p, int col0, int row, const WorkItem& it,
                                           uint32_t (&w)[4 * N]) {
    philox4x32_10<N>(static_cast<uint32_t>(col0) >> 3, static_cast<uint32_t>(row),
                     static_cast<uint32_t>(it.h), static_cast<uint32_t>(it.b), p.drop_seed_lo,
                     p.drop_seed_hi, w);
}

// Packs the probabilities of two adjacent keys for P V.  With dropout, a
// dropped one is packed as 0 (the caller's row sum keeps it); w is the word
// of drop_words that holds the pair's draws.
template <int FEAT, bool BF16>
__device__ __forceinline__ uint32_t pack_p(const FwdParams& p, float2 pp, uint32_t w) {
    if constexpr (FEAT == kDropout) {
        // low half >= t  <=>  (w << 16) >= (t << 16);  high half >= t  <=>  w >= (t << 16)
        return pack2<BF16>((w << 16) >= p.drop_threshold ? pp.x : 0.f,
                           w >= p.drop_threshold ? pp.y : 0.f);
    } else {
        return pack2<BF16>(pp.x, pp.y);
    }
}

// Issue the MMAs of S = Q K^T and of P V four K steps at a time, under one
// elect.sync (measured: b4h16 919 -> 945 TFLOP/s, D = 128 and the wide
// kernel unchanged within noise); 0 issues them one per election.
#ifndef FA_MMA_BATCH
#define FA_MMA_BATCH 1
#endif

template <int D, bool BF16, int NS, int RS, int FEAT>
__global__ void __launch_bounds__(Roles<RS>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
    using L = SmemLayout<D, NS, RS>;
    using R = Roles<RS>;
    constexpr int kRowSplit = RS;
    constexpr int kMmaWarp = R::kMmaWarp;
    constexpr int kLoadWarp = R::kLoadWarp;
    constexpr int kMmaWarp1 = R::kMmaWarp1;
    constexpr int kTileThreads = R::kTileThreads;
    constexpr int kChunks = D / 64;   // 128-byte column chunks per row (TMA box width)
    // Separate-P schedule (D = 64): P_t gets its own 64 TMEM columns, so S_t
    // of the next key tile can be computed as soon as the softmax has read
    // S_t into registers, while P_t V of this tile is still pending.
    // Otherwise P_t is written over S_t and the next S_t waits for P_t V
    // (same thread, in order).
    constexpr bool kSepP = separate_p(D);
    constexpr bool kMmaBatch = FA_MMA_BATCH != 0;
    constexpr bool kStageInQ = L::kStageInQ;
    constexpr bool kDirectO = L::kDirectO;
    constexpr int kPCol0 = kSepP ? (2 * kBN + 2 * D) : 0;   // P_0 column
    constexpr int kPColStride = kSepP ? (kBN / 2) : kBN;     // P_1 - P_0
    // Each of the kRowSplit threads of a row writes the packed P of its
    // kBN/kRowSplit keys as kBN/(2*kRowSplit) columns: contiguous in the
    // separate region, over the start of its own S columns otherwise.
    constexpr int kPHalfStride = kSepP ? (kBN / (2 * kRowSplit)) : (kBN / kRowSplit);
    constexpr int kStepsPerHalf = (kBN / kRowSplit) / 16;   // K=16 steps per half
    // TMEM column of the A operand (P_t) for K step kk of P_t V
    auto p_col = [](int t, int kk) {
        return kPCol0 + t * kPColStride + (kk / kStepsPerHalf) * kPHalfStride + (kk % kStepsPerHalf) * 8;
    };
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    Barriers<NS, RS>* bars = reinterpret_cast<Barriers<NS, RS>*>(smem + L::kOffBar);
    volatile int* abort_flag = &bars->abort;
    auto bar_addr = [&](const uint64_t* bptr) { return ptx::smem_addr(bptr); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Order of the K / V tiles of one item through the ring.  Aliased P:
    // K0 V0 K1 V1 ...  Separate P: K0 K1 V0 K2 V1 ... K(n-1) V(n-2) V(n-1),
    // since S_t(j+1) is issued before P_t(j) V_j.  The ring runs on across
    // items: an item's tiles follow the previous item's.
    auto ring_k = [](int j, int nkv) { return kSepP ? (j == 0 ? 0 : 2 * j - 1) : 2 * j; };
    auto ring_v = [](int j, int nkv) { return kSepP ? (j == nkv - 1 ? 2 * nkv - 1 : 2 * j + 2) : 2 * j + 1; };

    const uint32_t qbar = bar_addr(&bars->q_full);
    // ring position i of item `it` -> slot `slot`
    auto load_item = [&](const WorkItem& it, int i, int slot) {
        const uint32_t fb = bar_addr(&bars->kv_full[slot]);
        ptx::mbar_arrive_expect_tx(fb, L::kKVBytes);
        bool is_v;
        int j;
        if (!kSepP) {
            is_v = (i & 1) != 0;
            j = i >> 1;
        } else if (i == 0) {
            is_v = false;
            j = 0;
        } else if (i == 2 * it.nkv - 1) {
            is_v = true;
            j = it.nkv - 1;
        } else if (i & 1) {
            is_v = false;
            j = (i + 1) >> 1;
        } else {
            is_v = true;
            j = (i - 2) >> 1;
        }
        const CUtensorMap* m = is_v ? &tmV : &tmK;
        for (int c = 0; c < kChunks; ++c)
            ptx::tma_load_4d(sbase + L::kOffKV + slot * L::kKVBytes + c * (kBN * 128), m, fb, c * 64, it.hkv,
                             it.base + (it.jb + j) * kBN, it.tb);
    };
    // Q tiles of item `it` (a tile with no key tile is not loaded)
    auto load_q = [&](const WorkItem& it) {
        uint32_t qbytes = 0;
        for (int t = 0; t < kQTiles; ++t)
            if ((t == 0 ? it.nkv0 - it.s0 : it.nkv1 - it.s1) > 0) qbytes += L::kQBytes;
        ptx::mbar_arrive_expect_tx(qbar, qbytes);
        for (int t = 0; t < kQTiles; ++t) {
            if ((t == 0 ? it.nkv0 - it.s0 : it.nkv1 - it.s1) <= 0) continue;
            for (int c = 0; c < kChunks; ++c)
                ptx::tma_load_4d(sbase + L::kOffQ + t * L::kQBytes + c * (kBM * 128), &tmQ, qbar, c * 64,
                                 it.h, it.base + it.q0 + t * kBM, it.tb);
        }
    };

    // ---------------------------------------------------------------- setup
    // The producer thread initialises the barriers and starts the first
    // item's Q loads and the first round of its K / V ring before the
    // CTA-wide sync, so that their latency overlaps the TMEM allocation.
    int first_round = 0;   // ring items of the first item loaded before the sync
    if (warp == kLoadWarp && lane == 0) {
        // The kernel parameters are fixed before the launch: decode the first
        // item now, so that the latency of its parameter loads (cold right
        // after launch) overlaps the set-up and the wait for the previous
        // kernel.  Packed batches read their offsets from global memory,
        // which the previous kernel may still write: those decode after it.
        const int w_first = cta_item(0, p.items);
        WorkItem it_first{};
        if (FEAT != kPacked && w_first >= 0) it_first = decode_item<FEAT>(p, w_first);
        ptx::mbar_init(qbar, 1);
        ptx::mbar_init(bar_addr(&bars->q_empty), kQTiles);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(bar_addr(&bars->kv_full[s]), 1);
            ptx::mbar_init(bar_addr(&bars->kv_empty[s]), kSepP ? kQTiles : 1);   // one per MMA issuer
        }
        for (int t = 0; t < kQTiles; ++t) {
            ptx::mbar_init(bar_addr(&bars->s_full[t]), 1);
            ptx::mbar_init(bar_addr(&bars->s_free[t]), kTileThreads);
            ptx::mbar_init(bar_addr(&bars->p_full[t]), kTileThreads);
            ptx::mbar_init(bar_addr(&bars->p_half[t]), kTileThreads);
            ptx::mbar_init(bar_addr(&bars->o_done[t]), 1);
            ptx::mbar_init(bar_addr(&bars->drain[t]), 1);
        }
        bars->abort = 0;
        for (int d = 0; d < 7; ++d) bars->dbg[d] = 0;
        ptx::fence_barrier_init();
        ptx::tma_prefetch_map(&tmQ);
        ptx::tma_prefetch_map(&tmK);
        ptx::tma_prefetch_map(&tmV);
        ptx::tma_prefetch_map(&tmO);
        // Launched as a programmatic dependent of the previous kernel in the
        // stream, this CTA may have started before that kernel finished: it
        // reads and writes global memory only after this wait (everything
        // else in the CTA is ordered after it by the barriers and the sync).
        ptx::grid_dependency_wait();
        // this CTA's first item with key tiles (items of query blocks past the
        // end of a variable-length sequence have none)
        for (int k = 0;; ++k) {
            const int w = k == 0 ? w_first : cta_item(k, p.items);
            if (w < 0) break;
            const WorkItem it = (FEAT != kPacked && k == 0) ? it_first : decode_item<FEAT>(p, w);
            if (FEAT == kPacked && it.nkv == 0) continue;
            if (!p.drop_first_q) load_q(it);
            first_round = min(NS, 2 * it.nkv);
            for (int i = 0; i < first_round; ++i) load_item(it, i, i);
            break;
        }
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(&bars->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    debug_check((tmem & 0xffffu) == 0u);   // all 512 columns, from column 0
    // The next kernel in the stream (the combine launch of the split path, or
    // the next call) may be scheduled as soon as every CTA of this grid is
    // running; it waits for this grid to finish before touching memory.
    ptx::launch_dependents();

    // A bounded wait by every lane of a warp, with one outcome for the warp.
    auto wait_warp = [&](uint32_t bar, uint32_t parity, bool honour_abort = true) {
        return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, honour_abort));
    };

    // Each warpgroup changes its register budget with one instruction that
    // dominates all of its role code (ptxas allocates each region for it).
    if (warp >= kMmaWarp) {
        ptx::setmaxnreg_dec<R::kControlRegs>();
        if (warp == kLoadWarp) {
        // ------------------------------------------------------ TMA producer
        // The whole warp runs the loop and the waits; lane 0 issues the copies.
        {
            long long gi = 0;   // ring items issued, all items
            int k_q = 0;        // last item whose Q was loaded
            bool ok = true;
            // ring item gi goes to slot gi % NS once the item NS before it released it
            auto slot_free = [&](long long g) {
                return g < NS ||
                       wait_warp(bar_addr(&bars->kv_empty[g % NS]), static_cast<uint32_t>((g / NS - 1) & 1));
            };
            int ki = 0;   // items with key tiles so far (the barrier phases count these)
            for (int k = 0; ok; ++k) {
                const int w = cta_item(k, p.items);
                if (w < 0) break;
                const WorkItem it = decode_item<FEAT>(p, w);
                if (FEAT == kPacked && it.bad && lane == 0) atomicCAS(&g_fa_device_status, 0, kStatusBadSeqlens);
                if (FEAT == kPacked && it.nkv == 0) continue;
                const int n = 2 * it.nkv;
                int i = 0;
                if (ki == 0) {
                    // loaded before the sync, after the Q
                    i = __shfl_sync(0xffffffffu, first_round, 0);
                    gi = i;
                } else {
                    // With O staged in the Q buffer, the Q of this item waits
                    // for the previous item's epilogue: load the K / V tiles
                    // that only need free slots first.
                    const int pre = kStageInQ ? min(NS, n) : 0;
                    for (; i < pre; ++i, ++gi) {
                        if (!(ok = slot_free(gi))) break;
                        if (lane == 0) load_item(it, i, static_cast<int>(gi % NS));
                    }
                    if (!ok) break;
                    if (!(ok = wait_warp(bar_addr(&bars->q_empty), (ki - 1) & 1))) break;
                    if (lane == 0) load_q(it);
                    k_q = ki;
                }
                for (; i < n; ++i, ++gi) {
                    if (!(ok = slot_free(gi))) break;
                    if (lane == 0) load_item(it, i, static_cast<int>(gi % NS));
                }
                ++ki;
            }
            if (FA_DEBUG && lane == 0) bars->dbg[0] = static_cast<int>(gi);
            if (*abort_flag) {
                // Let every copy this warp started land before the CTA exits.
                wait_warp(qbar, k_q & 1, false);
                for (long long i = (gi > NS ? gi - NS : 0); i < gi; ++i)
                    wait_warp(bar_addr(&bars->kv_full[i % NS]), static_cast<uint32_t>((i / NS) & 1), false);
            }
        }
    } else if (kSepP && (warp == kMmaWarp || warp == kMmaWarp1)) {
        // ------------------------------------------- MMA issuers (separate P)
        // One issuing warp per query tile, so that each tile's products wait
        // only on its own softmax; the whole warp runs the loop and one
        // elected lane issues the MMAs and commits.  Both issuers see every K / V tile of
        // the ring in the same order and release each slot once (a commit
        // after the products that read it, or a plain arrive once it has
        // landed when this tile has no work on it), and each releases the Q
        // buffer of an item once its last S_t has been computed.
        {
            const int t = (warp == kMmaWarp) ? 0 : 1;
            constexpr uint32_t kIdescQK = ptx::idesc_f16_f32(kBM, kBN, BF16, false);
            constexpr uint32_t kIdescPV = ptx::idesc_f16_f32(kBM, D, BF16, true);
            // ring positions are kept modulo 2*NS: slot and phase parity only
            auto full_bar = [&](int i) { return bar_addr(&bars->kv_full[i % NS]); };
            auto full_par = [&](int i) { return static_cast<uint32_t>((i / NS) & 1); };
            auto slot_addr = [&](int i) { return sbase + L::kOffKV + (i % NS) * L::kKVBytes; };
            const uint32_t s_full = bar_addr(&bars->s_full[t]);
            const uint32_t s_free = bar_addr(&bars->s_free[t]);
            const uint32_t p_full = bar_addr(&bars->p_full[t]);
            const uint32_t o_done = bar_addr(&bars->o_done[t]);
            const uint32_t q_empty = bar_addr(&bars->q_empty);

            // S_t = Q_t K^T over D in K=16 steps; both operands K-major.
            auto issue_s = [&](int ring) {
                if constexpr (kMmaBatch) {
                    // four K steps per election; 128-byte column chunks of
                    // Q and K are kBM*128 and kBN*128 bytes apart
                    const uint32_t hi = ptx::sdesc_sw128_hi(1024);
                    const uint32_t a0 = ptx::sdesc_sw128_lo(sbase + L::kOffQ + t * L::kQBytes, 16);
                    const uint32_t b0 = ptx::sdesc_sw128_lo(slot_addr(ring), 16);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        ptx::mma_ss_x4_lo(tmem + t * kBN, a0 + c * (kBM * 128 / 16), b0 + c * (kBN * 128 / 16), hi,
                                          2u, kIdescQK, c > 0 ? 1u : 0u);
                } else {
                    const uint64_t a0 = ptx::sdesc_sw128(sbase + L::kOffQ + t * L::kQBytes, 16, 1024);
                    const uint64_t b0 = ptx::sdesc_sw128(slot_addr(ring), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t oa = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
                        const uint32_t ob = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
                        ptx::mma_ss_warp(tmem + t * kBN, a0 + (oa >> 4), b0 + (ob >> 4), kIdescQK, kk > 0);
                    }
                }
                ptx::tc_commit_warp(s_full);
                ptx::tc_commit_warp(bar_addr(&bars->kv_empty[ring % NS]));
            };
            // O_t (+)= P_t V over the keys [kk0*16, kk1*16) of the tile in
            // K=16 steps; P from TMEM, V MN-major (64-column chunks kBN*128
            // bytes apart).
            auto issue_pv = [&](int ring, bool acc, int kk0, int kk1) {
                if constexpr (kMmaBatch) {
                    static_assert(kBN / 32 == 4, "P V halves of four K steps");
                    // P columns of consecutive K steps are 8 apart, V rows
                    // 16 keys x 128 bytes
                    const uint32_t hi = ptx::sdesc_sw128_hi(1024);
                    const uint32_t b0 = ptx::sdesc_sw128_lo(slot_addr(ring), kBN * 128);
                    ptx::mma_ts_x4_lo(tmem + 2 * kBN + t * D, tmem + p_col(t, kk0), b0 + kk0 * (16 * 128 / 16), hi,
                                      8u, 16u * 128u / 16u, kIdescPV, (acc || kk0 > 0) ? 1u : 0u);
                } else {
                    const uint64_t b0 = ptx::sdesc_sw128(slot_addr(ring), kBN * 128, 1024);
#pragma unroll
                    for (int kk = kk0; kk < kk1; ++kk) {
                        ptx::mma_ts_warp(tmem + 2 * kBN + t * D, tmem + p_col(t, kk),
                                         b0 + ((kk * 16 * 128) >> 4), kIdescPV, (acc || kk > 0) ? 1u : 0u);
                    }
                }
            };
            // wait for item `ring` to land; release it at once when `use` is false
            auto acquire = [&](int ring, bool use) {
                if (!wait_warp(full_bar(ring), full_par(ring))) return false;
                if (use) ptx::tc_fence_after_sync();
                else ptx::mbar_arrive_warp(bar_addr(&bars->kv_empty[ring % NS]));
                return true;
            };

            int gi0 = 0;       // ring position of the item's first tile, modulo 2*NS
            int ring_total = 0;   // ring items seen, all items (FA_DEBUG count)
            uint32_t gs = 0;   // S_t tiles issued, all items (parities only)
            bool ok = true;
            int ki = 0;   // items with key tiles so far
            for (int k = 0; ok; ++k) {
                const int w = cta_item(k, p.items);
                if (w < 0) break;
                const WorkItem it = decode_item<FEAT>(p, w);
                if (FEAT == kPacked && it.nkv == 0) continue;
                const int nkv = it.nkv;
                const int s_t = FEAT != kLocal ? 0 : (t == 0) ? it.s0 : it.s1;    // key tiles [s_t, n_t)
                const int n_t = (t == 0) ? it.nkv0 : it.nkv1;
                auto used = [&](int j) { return j >= s_t && j < n_t; };
                const uint32_t gs0 = gs;   // S_t / P_t / P_t V index of this tile's first key tile
                // every issuer waits for every Q load, so that its phases stay in step
                if (!(ok = wait_warp(qbar, ki & 1))) break;
                ++ki;
                if (!(ok = acquire(gi0 + ring_k(0, nkv), used(0)))) break;
                if (used(0)) {
                    // S_t of the previous item must have been read by the softmax
                    if (gs > 0 && !(ok = wait_warp(s_free, (gs - 1) & 1))) break;
                    ptx::tc_fence_after_sync();
                    issue_s(gi0 + ring_k(0, nkv));
                    ++gs;
                }
                // the Q buffer of tile t is free once its last S_t is complete
                if (n_t <= s_t) ptx::mbar_arrive_warp(q_empty);
                else if (n_t == 1) ptx::tc_commit_warp(q_empty);
                for (int j = 0; ok && j < nkv; ++j) {
                    // S_t(j+1) as soon as the softmax holds S_t(j), then P_t V(j)
                    if (j + 1 < nkv) {
                        const bool use = used(j + 1);
                        if (!(ok = acquire(gi0 + ring_k(j + 1, nkv), use))) break;
                        if (use) {
                            if (gs > 0 && !(ok = wait_warp(s_free, (gs - 1) & 1))) break;
                            ptx::tc_fence_after_sync();
                            issue_s(gi0 + ring_k(j + 1, nkv));
                            ++gs;
                            if (j + 2 == n_t) ptx::tc_commit_warp(q_empty);
                        }
                    }
                    if (!(ok = acquire(gi0 + ring_v(j, nkv), used(j)))) break;
                    if (used(j)) {
                        // P_t V(j) in two halves: the first 64 keys as soon as
                        // the softmax has stored their P (and rescaled O_t if it
                        // had to), the rest once all of P_t(j) is written.  This
                        // also orders the item's first P_t V after the previous
                        // epilogue's reads of O_t.
                        const int ring = gi0 + ring_v(j, nkv);
                        const uint32_t g = gs0 + static_cast<uint32_t>(j - s_t);
                        if (!(ok = wait_warp(bar_addr(&bars->p_half[t]), g & 1))) break;
                        ptx::tc_fence_after_sync();
                        issue_pv(ring, j > s_t, 0, kBN / 32);
                        if (!(ok = wait_warp(p_full, g & 1))) break;
                        ptx::tc_fence_after_sync();
                        issue_pv(ring, true, kBN / 32, kBN / 16);
                        ptx::tc_commit_warp(o_done);
                        ptx::tc_commit_warp(bar_addr(&bars->kv_empty[ring % NS]));
                    }
                }
                gi0 = (gi0 + 2 * nkv) % (2 * NS);
                ring_total += 2 * nkv;
            }
            if (FA_DEBUG && lane == 0) {
                bars->dbg[1 + t] = ring_total;
                bars->dbg[3 + t] = static_cast<int>(gs);
            }
            // Every MMA of this issuer must be complete before TMEM is freed.
            ptx::tc_commit_warp(bar_addr(&bars->drain[t]));
            wait_warp(bar_addr(&bars->drain[t]), 0, false);
        }
    } else if (!kSepP && warp == kMmaWarp) {
        // ----------------------------------------------- MMA issuer (P over S)
        // One warp (one elected lane issuing) runs both tiles' products in
        // the order
        //   S0(0) S1(0) | P0V(j) S0(j+1) P1V(j) S1(j+1) | ...
        // so that one tile's softmax runs while the other tile's products do;
        // S_t(j+1) follows P_t V(j), which reads the P_t it overwrites.  The
        // next item's S_t(0) follows this item's last P_t V the same way.
        {
            constexpr uint32_t kIdescQK = ptx::idesc_f16_f32(kBM, kBN, BF16, false);
            constexpr uint32_t kIdescPV = ptx::idesc_f16_f32(kBM, D, BF16, true);
            auto full_bar = [&](int i) { return bar_addr(&bars->kv_full[i % NS]); };
            auto full_par = [&](int i) { return static_cast<uint32_t>((i / NS) & 1); };
            auto slot_addr = [&](int i) { return sbase + L::kOffKV + (i % NS) * L::kKVBytes; };
            // descriptors as low words over one shared high word (SBO 1024,
            // 128-byte swizzle); the start address field counts 16 bytes
            const uint32_t desc_hi = ptx::sdesc_sw128_hi(1024);
            auto issue_s = [&](int t, int ring) {
                const uint32_t a0 = ptx::sdesc_sw128_lo(sbase + L::kOffQ + t * L::kQBytes, 16);
                const uint32_t b0 = ptx::sdesc_sw128_lo(slot_addr(ring), 16);
                if constexpr (kMmaBatch) {
                    // four K steps (one 128-byte column chunk) per election
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        ptx::mma_ss_x4_lo(tmem + t * kBN, a0 + c * (kBM * 128 / 16), b0 + c * (kBN * 128 / 16),
                                          desc_hi, 2u, kIdescQK, c > 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t oa = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
                        const uint32_t ob = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
                        ptx::mma_ss_warp_lo(tmem + t * kBN, a0 + (oa >> 4), b0 + (ob >> 4), desc_hi, kIdescQK,
                                            kk > 0);
                    }
                }
                ptx::tc_commit_warp(bar_addr(&bars->s_full[t]));
            };
            auto issue_pv = [&](int t, int ring, bool acc) {
                const uint32_t b0 = ptx::sdesc_sw128_lo(slot_addr(ring), kBN * 128);
                if constexpr (kMmaBatch) {
                    // four K steps per election; P columns of consecutive steps
                    // are 8 apart within each of the RS column blocks
                    static_assert(kStepsPerHalf % 4 == 0, "P V in runs of four K steps");
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; kk += 4)
                        ptx::mma_ts_x4_lo(tmem + 2 * kBN + t * D, tmem + p_col(t, kk), b0 + kk * (16 * 128 / 16),
                                          desc_hi, 8u, 16u * 128u / 16u, kIdescPV, (acc || kk > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        ptx::mma_ts_warp_lo(tmem + 2 * kBN + t * D, tmem + p_col(t, kk), b0 + ((kk * 16 * 128) >> 4),
                                            desc_hi, kIdescPV, (acc || kk > 0) ? 1u : 0u);
                    }
                }
                ptx::tc_commit_warp(bar_addr(&bars->o_done[t]));
            };

            int gi0 = 0;                   // ring position of the item's K0, modulo 2*NS
            int ring_total = 0;            // ring items seen, all items (FA_DEBUG count)
            uint32_t gs[kQTiles] = {0, 0};  // S_t tiles issued per query tile (parities only)
            bool ok = true;
            int ki = 0;   // items with key tiles so far
            for (int k = 0; ok; ++k) {
                const int w = cta_item(k, p.items);
                if (w < 0) break;
                const WorkItem it = decode_item<FEAT>(p, w);
                if (FEAT == kPacked && it.nkv == 0) continue;
                const int nkv = it.nkv, nkv0 = it.nkv0, nkv1 = it.nkv1;
                const int s0 = FEAT == kLocal ? it.s0 : 0, s1 = FEAT == kLocal ? it.s1 : 0;
                const uint32_t g00 = gs[0], g10 = gs[1];
                if (!(ok = wait_warp(qbar, ki & 1))) break;
                ++ki;
                // with O stored directly, the Q buffer of tile t is free once
                // its last S_t is complete (a tile without keys: now, after
                // this item's Q load)
                const uint32_t q_empty = bar_addr(&bars->q_empty);
                if (kDirectO && nkv0 <= s0) ptx::mbar_arrive_warp(q_empty);
                if (kDirectO && nkv1 <= s1) ptx::mbar_arrive_warp(q_empty);
                const int k0 = gi0 + ring_k(0, nkv);
                if (!(ok = wait_warp(full_bar(k0), full_par(k0)))) break;
                ptx::tc_fence_after_sync();
                if (s0 == 0 && nkv0 > 0) {
                    issue_s(0, k0);
                    if (kDirectO && nkv0 == 1) ptx::tc_commit_warp(q_empty);
                }
                if (s1 == 0 && nkv1 > 0) {
                    issue_s(1, k0);
                    if (kDirectO && nkv1 == 1) ptx::tc_commit_warp(q_empty);
                }
                ptx::tc_commit_warp(bar_addr(&bars->kv_empty[k0 % NS]));
                for (int j = 0; ok && j < nkv; ++j) {
                    const int iv = gi0 + ring_v(j, nkv);
                    const int ik = gi0 + ring_k(j + 1, nkv);
                    const bool next = (j + 1) < nkv;
                    if (!(ok = wait_warp(full_bar(iv), full_par(iv)))) break;
                    ptx::tc_fence_after_sync();
                    if (j >= s0 && j < nkv0) {
                        if (!(ok = wait_warp(bar_addr(&bars->p_full[0]), (g00 + j - s0) & 1))) break;
                        ptx::tc_fence_after_sync();
                        issue_pv(0, iv, j > s0);
                    }
                    if (next) {
                        if (!(ok = wait_warp(full_bar(ik), full_par(ik)))) break;
                        ptx::tc_fence_after_sync();
                    }
                    if (j + 1 >= s0 && j + 1 < nkv0) {
                        issue_s(0, ik);
                        if (kDirectO && j + 2 == nkv0) ptx::tc_commit_warp(q_empty);
                    }
                    if (j >= s1 && j < nkv1) {
                        if (!(ok = wait_warp(bar_addr(&bars->p_full[1]), (g10 + j - s1) & 1))) break;
                        ptx::tc_fence_after_sync();
                        issue_pv(1, iv, j > s1);
                    }
                    ptx::tc_commit_warp(bar_addr(&bars->kv_empty[iv % NS]));
                    if (j + 1 >= s1 && j + 1 < nkv1) {
                        issue_s(1, ik);
                        if (kDirectO && j + 2 == nkv1) ptx::tc_commit_warp(q_empty);
                    }
                    if (next) ptx::tc_commit_warp(bar_addr(&bars->kv_empty[ik % NS]));
                }
                gs[0] += max(0, nkv0 - s0);
                gs[1] += max(0, nkv1 - s1);
                gi0 = (gi0 + 2 * nkv) % (2 * NS);
                ring_total += 2 * nkv;
            }
            if (FA_DEBUG && lane == 0) {
                bars->dbg[1] = bars->dbg[2] = ring_total;
                bars->dbg[3] = static_cast<int>(gs[0]);
                bars->dbg[4] = static_cast<int>(gs[1]);
            }
            // Every MMA must be complete before TMEM is freed.
            ptx::tc_commit_warp(bar_addr(&bars->drain[0]));
            wait_warp(bar_addr(&bars->drain[0]), 0, false);
        }
    }
    } else {
        ptx::setmaxnreg_inc<R::kSoftmaxRegs>();
        // ----------------------------------------------------- softmax groups
        // Warp w works on query tile t = w / (4 RS), score columns
        // [hf*128/RS, (hf+1)*128/RS) of each key tile (hf = (w / 4) % RS),
        // rows 32*wq .. 32*wq+31 of the tile (wq = w % 4, the TMEM lane
        // quarter it may access).  With RS = 2 the two threads of a row swap
        // their partial maxima every key tile, so both keep the same reference
        // max; each keeps its own partial row sum.  After an abort every warp
        // still walks every item and runs every named barrier (with no TMEM
        // work), so the barriers cannot hang.
        constexpr int kHalf = kBN / kRowSplit;      // score columns per thread
        constexpr int kDH = D / kRowSplit;          // O columns per thread
        const int t = warp / (4 * kRowSplit);
        const int hf = (warp >> 2) % kRowSplit;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;               // row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * kBN + hf * kHalf;
        const uint32_t tO = tmem + lane_off + 2 * kBN + t * D + hf * kDH;
        // P: kHalf/2 packed columns per thread, in the separate P region or
        // over the first kHalf/2 columns of this thread's own part of S_t
        const uint32_t tP = tmem + lane_off +
                            (kSepP ? (kPCol0 + t * kPColStride + hf * (kHalf / 2)) : (t * kBN + hf * kHalf));
        const uint32_t pair_bar = 1 + t * 4 + wq;   // the RS warps sharing these rows
        const uint32_t tile_bar = 1 + 4 * kQTiles + t;
        const bool store_thread = (r == 0 && hf == 0);   // issues this tile's O stores
        const float c = p.scale_log2;
        // After an abort, one thread per row simply leaves the key loop; with
        // the row split, a warp keeps running its loop without TMEM stores or
        // arrivals instead, so that the swap barriers stay matched.
        constexpr bool kBreakOnAbort = (kRowSplit == 1);
        bool ok = true;
        uint32_t gs0 = 0;   // S_t tiles of earlier items (parities only)

        int ki = 0;   // items with key tiles so far (the barrier phases count these)
        for (int k = 0;; ++k) {
            const int w = cta_item(k, p.items);
            if (w < 0) break;
            const WorkItem it = decode_item<FEAT>(p, w);
            if (FEAT == kPacked && it.nkv == 0) continue;
            const int r0 = it.q0 + t * kBM;
            const int row = r0 + r;
            const int s_t = FEAT != kLocal ? 0 : (t == 0) ? it.s0 : it.s1;
            const int n_tiles = max(0, ((t == 0) ? it.nkv0 : it.nkv1) - s_t);   // key tiles of this tile

            float m_use = -INFINITY;   // reference max, raw (unscaled) score units
            float l = 0.f;             // this thread's part of the row sum
            bool use_max_next = false; // the previous tile moved the reference
            for (int j = 0; j < n_tiles; ++j) {
                ok = (kBreakOnAbort || ok) && wait_phase(bar_addr(&bars->s_full[t]), (gs0 + j) & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (kBreakOnAbort && !ok) break;
                ptx::tc_fence_after_sync();
                uint32_t s[kHalf];
                const int kv0 = (it.jb + s_t + j) * kBN + hf * kHalf;   // key of column 0
                // Keys past the end and, on diagonal tiles, keys after the row are masked.
                float alpha = 1.f;
                bool rescale = false;
                if constexpr (kRowSplit == 1) {
                    // keys outside [first, last] are masked: past the sequence,
                    // after the row (causal) or outside the window
                    const bool need_mask = kv0 + kHalf > it.S || (p.causal && kv0 + kHalf - 1 > r0) ||
                                           (FEAT == kLocal && p.win_left >= 0 && kv0 < r0 + kBM - 1 - p.win_left) ||
                                           (FEAT == kLocal && p.win_right >= 0 && kv0 + kHalf - 1 > r0 + p.win_right);
                    int last = p.causal ? min(it.S - 1, row) : (it.S - 1);
                    if (FEAT == kLocal && p.win_right >= 0) last = min(last, row + p.win_right);
                    const int first = (FEAT == kLocal && p.win_left >= 0) ? row - p.win_left : -1;
                    constexpr int kChains = 4;
                    float mx[kChains];
#pragma unroll
                    for (int i = 0; i < kChains; ++i) mx[i] = -INFINITY;
                    auto mask_max = [&](int k0, int k1) {
                        if (need_mask) {
#pragma unroll
                            for (int kq = k0; kq < k1; ++kq)
                                if (kv0 + kq > last || (FEAT == kLocal && kv0 + kq < first)) s[kq] = __float_as_uint(-INFINITY);
                        }
#pragma unroll
                        for (int kq = k0 / 2; kq < k1 / 2; ++kq)
                            mx[kq % kChains] = ptx::fmax3(mx[kq % kChains], __uint_as_float(s[2 * kq]),
                                                          __uint_as_float(s[2 * kq + 1]));
                    };
#pragma unroll
                    for (int q = 0; q < kHalf / 32; ++q) ptx::tmem_ld_32x32b_x32(tS + q * 32, s + q * 32);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence<kHalf>(s);
                    if (kSepP && (kBreakOnAbort || ok)) {
                        // S_t is in registers: the next S_t may overwrite it
                        ptx::tc_fence_before_sync();
                        ptx::mbar_arrive(bar_addr(&bars->s_free[t]));
                    }
                    mask_max(0, kHalf);
                    float m_tile = mx[0];
#pragma unroll
                    for (int i = 1; i < kChains; ++i) m_tile = fmaxf(m_tile, mx[i]);
                    if constexpr (kRowSplit > 1) {
                        bars->row_max[j & 1][t][hf][r] = m_tile;
                        ptx::named_barrier_sync(pair_bar, 32 * kRowSplit);
                        m_tile = fmaxf(m_tile, bars->row_max[j & 1][t][hf ^ 1][r]);
                    }
                    const float m_new = fmaxf(m_use, m_tile);
                    // Lazy rescale: keep the old reference unless the max grew by more
                    // than kTauLog2 in log2 units (then p <= 2^kTauLog2).  The RS
                    // threads of a row see the same maxima, so they decide alike.
                    rescale = (m_new - m_use) * c > kTauLog2;
                    if (rescale) {
                        alpha = ptx::ex2_approx((m_use - m_new) * c);
                        m_use = m_new;
                    }
                    const float mc = (m_use == -INFINITY) ? 0.f : m_use * c;

                    // p = 2^(s*c - m*c), two columns per packed FMA / add
                    const float2 c2 = make_float2(c, c);
                    const float2 nmc2 = make_float2(-mc, -mc);
                    float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                    for (int q = 0; q < kHalf / 32; ++q) {
                        uint32_t pk[16];
                        uint32_t dw[16] = {};   // dropout draws of these 32 keys
                        if constexpr (FEAT == kDropout) drop_words<4>(p, kv0 + q * 32, row, it, dw);
#pragma unroll
                        for (int kq = 0; kq < 16; ++kq) {
                            const float2 x = __ffma2_rn(
                                make_float2(__uint_as_float(s[q * 32 + 2 * kq]),
                                            __uint_as_float(s[q * 32 + 2 * kq + 1])),
                                c2, nmc2);
                            const float2 pp = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
                            sum2[kq & 1] = __fadd2_rn(sum2[kq & 1], pp);
                            pk[kq] = pack_p<FEAT, BF16>(p, pp, dw[kq]);
                        }
                        if (kSepP && q == 0 && j > 0 && ok) {
                            // P_t and O_t are still read / written by P_t V of tile j-1
                            ok = wait_phase(bar_addr(&bars->o_done[t]), (gs0 + j - 1) & 1, abort_flag);
                            ok = __all_sync(0xffffffffu, ok);
                            if (kBreakOnAbort && !ok) break;
                            ptx::tc_fence_after_sync();
                            // O_t is rescaled before any of P_t V(j) can start
                            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                                for (int q2 = 0; q2 < kDH / 32; ++q2) {
                                    uint32_t o[32];
                                    ptx::tmem_ld_32x32b_x32(tO + q2 * 32, o);
                                    ptx::tmem_ld_wait();
                                    ptx::reg_fence<32>(o);
#pragma unroll
                                    for (int u = 0; u < 32; ++u)
                                        o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
                                    ptx::tmem_st_32x32b_x32(tO + q2 * 32, o);
                                }
                            }
                        }
                        if (kBreakOnAbort || ok) ptx::tmem_st_32x32b_x16(tP + q * 16, pk);
                        if (kSepP && q == (kHalf / 32) / 2 - 1 && (kBreakOnAbort || ok)) {
                            // the first half of P_t(j) may be read
                            ptx::tmem_st_wait();
                            ptx::tc_fence_before_sync();
                            ptx::mbar_arrive(bar_addr(&bars->p_half[t]));
                        }
                    }
                    if (kBreakOnAbort && !ok) break;
                    const float2 sum = __fadd2_rn(sum2[0], sum2[1]);
                    l = l * alpha + (sum.x + sum.y);
                } else {
                    // keys outside [first, last] are masked: past the sequence,
                    // after the row (causal) or outside the window
                    const bool need_mask = kv0 + kHalf > it.S || (p.causal && kv0 + kHalf - 1 > r0) ||
                                           (FEAT == kLocal && p.win_left >= 0 && kv0 < r0 + kBM - 1 - p.win_left) ||
                                           (FEAT == kLocal && p.win_right >= 0 && kv0 + kHalf - 1 > r0 + p.win_right);
                    int last = p.causal ? min(it.S - 1, row) : (it.S - 1);
                    if (FEAT == kLocal && p.win_right >= 0) last = min(last, row + p.win_right);
                    const int first = (FEAT == kLocal && p.win_left >= 0) ? row - p.win_left : -1;
#pragma unroll
                    for (int q = 0; q < kHalf / 32; ++q) ptx::tmem_ld_32x32b_x32(tS + q * 32, s + q * 32);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence<kHalf>(s);
                    if (kSepP && (kBreakOnAbort || ok)) {
                        // S_t is in registers: the next S_t may overwrite it
                        ptx::tc_fence_before_sync();
                        ptx::mbar_arrive(bar_addr(&bars->s_free[t]));
                    }
                    if (need_mask) {
#pragma unroll
                        for (int kq = 0; kq < kHalf; ++kq)
                            if (kv0 + kq > last || (FEAT == kLocal && kv0 + kq < first)) s[kq] = __float_as_uint(-INFINITY);
                    }

                    // One pass over this thread's columns: p = 2^(s*c - mc), two
                    // columns per packed FMA / add, written to TMEM as packed 16-bit
                    // P (with separate P, once P_t V of tile j-1 has released P_t).
                    bool p_free = !(kSepP && j > 0);
                    float sum = 0.f;
                    auto exp_pass = [&](float mc) {
                        const float2 c2 = make_float2(c, c);
                        const float2 nmc2 = make_float2(-mc, -mc);
                        float2 sum2[1] = {make_float2(0.f, 0.f)};
                        // 16 columns at a time (registers are short with two
                        // threads per row)
#pragma unroll
                        for (int q = 0; q < kHalf / 16; ++q) {
                            uint32_t pk[8];
                            uint32_t dw[4] = {};   // dropout draws of 8 of these keys
#pragma unroll
                            for (int kq = 0; kq < 8; ++kq) {
                                const float2 x = __ffma2_rn(
                                    make_float2(__uint_as_float(s[q * 16 + 2 * kq]),
                                                __uint_as_float(s[q * 16 + 2 * kq + 1])),
                                    c2, nmc2);
                                const float2 pp = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
                                sum2[0] = __fadd2_rn(sum2[0], pp);
                                // (one block at a time: two threads share a row here
                                // and registers are short)
                                if constexpr (FEAT == kDropout)
                                    if ((kq & 3) == 0) drop_words<1>(p, kv0 + q * 16 + 2 * kq, row, it, dw);
                                pk[kq] = pack_p<FEAT, BF16>(p, pp, dw[kq & 3]);
                            }
                            if (!p_free && ok) {
                                // P_t and O_t are still read / written by P_t V of tile j-1
                                ok = wait_phase(bar_addr(&bars->o_done[t]), (gs0 + j - 1) & 1, abort_flag);
                                ok = __all_sync(0xffffffffu, ok);
                                if (ok) ptx::tc_fence_after_sync();
                                p_free = true;
                            }
                            if (ok) ptx::tmem_st_32x32b_x8(tP + q * 8, pk);
                        }
                        sum = sum2[0].x + sum2[0].y;
                    };

                    // this tile's row max (the RS threads of a row swap their parts)
                    auto tile_max = [&]() {
                        constexpr int kChains = 4;
                        float mx[kChains];
#pragma unroll
                        for (int i = 0; i < kChains; ++i) mx[i] = -INFINITY;
#pragma unroll
                        for (int kq = 0; kq < kHalf / 2; ++kq)
                            mx[kq % kChains] = ptx::fmax3(mx[kq % kChains], __uint_as_float(s[2 * kq]),
                                                          __uint_as_float(s[2 * kq + 1]));
                        float m_tile = mx[0];
#pragma unroll
                        for (int i = 1; i < kChains; ++i) m_tile = fmaxf(m_tile, mx[i]);
                        if constexpr (kRowSplit > 1) {
                            bars->row_max[j & 1][t][hf][r] = m_tile;
                            ptx::named_barrier_sync(pair_bar, 32 * kRowSplit);
                            m_tile = fmaxf(m_tile, bars->row_max[j & 1][t][hf ^ 1][r]);
                        }
                        return m_tile;
                    };
                    {
                        // With the row split the two threads of a row would swap
                        // their maxima every tile.  Instead the exponentials are
                        // first taken against the current reference: the lazy
                        // rescale only has to move it when some p would exceed
                        // 2^kTauLog2, and the row sum (p >= 0) bounds every p, so a
                        // sum <= 2^kTauLog2 keeps the reference.  Otherwise (an
                        // item's first tile, a failed check, or a previous tile that
                        // moved the reference) the tile max comes first and the
                        // reference moves up to it.  TMEM stores are warp-wide and
                        // the two threads of a row share its reference, so the pair
                        // of warps on these rows takes one path.
                        // (a row with no key yet -- the first tile, or a window
                        // that has not reached its keys -- has no reference: a
                        // warp-wide choice, like everything that feeds the named
                        // barriers and TMEM stores below)
                        bool with_max = __any_sync(0xffffffffu, m_use == -INFINITY) || use_max_next;
                        if (!with_max) {
                            exp_pass(m_use * c);
                            with_max = ptx::named_barrier_or(pair_bar, 32 * kRowSplit,
                                                             !(sum <= kMaxTileSum));   // also inf / NaN
                            if (with_max) ptx::tmem_st_wait();   // these P stores land first
                        }
                        if (with_max) {
                            const float m_tile = tile_max();
                            if (m_tile > m_use) {
                                alpha = ptx::ex2_approx((m_use - m_tile) * c);   // 0 on the first tile
                                m_use = m_tile;
                                rescale = true;
                            }
                            exp_pass(m_use == -INFINITY ? 0.f : m_use * c);
                        }
                        // peaky scores keep raising the max: take it first next time
                        // (both warps of the pair cover the same rows: same choice)
                        use_max_next = __any_sync(0xffffffffu, rescale && j > 0);
                    }
                    if (kBreakOnAbort && !ok) break;
                    l = l * alpha + sum;
                }

                // O_t was last written by P V of tile j-1: with separate P its
                // completion was awaited above; with P over S it completed before
                // S_t of tile j (same issuing thread, in order).
                if ((kBreakOnAbort || ok) && j > 0 && !(kSepP && kRowSplit == 1) &&
                    __any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int q = 0; q < kDH / 32; ++q) {
                        uint32_t o[32];
                        ptx::tmem_ld_32x32b_x32(tO + q * 32, o);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence<32>(o);
#pragma unroll
                        for (int kq = 0; kq < 32; ++kq) o[kq] = __float_as_uint(__uint_as_float(o[kq]) * alpha);
                        ptx::tmem_st_32x32b_x32(tO + q * 32, o);
                    }
                }
                if (kBreakOnAbort || ok) {
                    ptx::tmem_st_wait();
                    ptx::tc_fence_before_sync();
                    // with the row split all of P_t is released at once
                    if (kSepP && kRowSplit > 1) ptx::mbar_arrive(bar_addr(&bars->p_half[t]));
                    ptx::mbar_arrive(bar_addr(&bars->p_full[t]));
                }
            }

            // With two threads per row registers are short: the epilogue
            // decodes its item again instead of keeping these fields live
            // through the key loop (the opaque copy of w stops the compiler
            // from reusing the first decode).  Packed batches read their
            // offsets from global memory, so they keep the first decode.
            const WorkItem ie = (kRowSplit > 1 && FEAT != kPacked) ? decode_item<FEAT>(p, ptx::opaque(w)) : it;
            // ------------------------------------------------------- epilogue
            // O_t is read out of TMEM (and waited for) before this thread's first
            // P_t arrival of the next item, which the next item's first P_t V
            // awaits: that orders its overwrite of O_t after these reads.
            bool eok = ok;
            if (n_tiles > 0)
                eok = eok && wait_phase(bar_addr(&bars->o_done[t]), (gs0 + n_tiles - 1) & 1, abort_flag);
            eok = __all_sync(0xffffffffu, eok);
            // whole-row sum from the RS parts
            float l_row = l;
            if constexpr (kRowSplit > 1) {
                bars->row_sum[ki & 1][t][hf][r] = l;
                ptx::named_barrier_sync(pair_bar, 32 * kRowSplit);
                l_row = l + bars->row_sum[ki & 1][t][hf ^ 1][r];
            }
            // With O staged in the Q buffer, this tile's store thread frees
            // the buffer for the next item's Q.  A tile with no key tile has
            // no product that orders its release after this item's Q load:
            // it waits for that load first, so that the release counts for
            // this item and not for the previous one.
            auto release_q = [&]() {
                if (n_tiles == 0 && !wait_phase(qbar, ki & 1, abort_flag)) return;
                ptx::mbar_arrive(bar_addr(&bars->q_empty));
            };
            if (ie.partial && r0 < ie.S) {
                // partial result: o~ stays unnormalised (fp32), m and l go
                // beside it; a tile that saw no key of this split records l = 0
                const int ntq = (p.S + kBM - 1) / kBM;
                const size_t slot = partial_slot(ie.bh, ntq, r0 / kBM, p.max_splits, ie.split);
                float* ml = p.ws_ml + slot * (2 * kBM);
                float4* po = reinterpret_cast<float4*>(p.ws_o + slot * static_cast<size_t>(kBM * D));
                if (eok && n_tiles > 0) {
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int q = 0; q < kDH / 32; ++q) {
                        uint32_t o[32];
                        ptx::tmem_ld_32x32b_x32(tO + q * 32, o);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence<32>(o);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            po[(hf * (kDH / 4) + q * 8 + u) * kBM + r] =
                                make_float4(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1]),
                                            __uint_as_float(o[4 * u + 2]), __uint_as_float(o[4 * u + 3]));
                    }
                    if (hf == 0) {
                        ml[r] = m_use * c;
                        ml[kBM + r] = l_row;
                    }
                } else if (eok && hf == 0) {
                    ml[r] = -INFINITY;
                    ml[kBM + r] = 0.f;
                }
                if (kStageInQ && eok && store_thread) release_q();
            } else if (n_tiles > 0) {
                // final result: stage O_t as the 128-byte-swizzled TMA box, then
                // one thread stores it; rows past S are dropped by the store.
                // The last tile of a packed sequence is stored row by row
                // instead (the rows after it belong to the next sequence).
                const bool direct = kDirectO || (FEAT == kPacked && r0 + kBM > ie.S);
                uint8_t* stage = smem + L::kOffStage + t * L::kQBytes;
                if (!kStageInQ && !direct && ki > 0) {
                    // the previous item's store must have read the staging buffer
                    if (store_thread) ptx::bulk_wait_group_read_all();
                    ptx::named_barrier_sync(tile_bar, kTileThreads);
                }
                // a stored row saw at least one key (its own, or key 0)
                if (eok && row < ie.S) debug_check(l_row > 0.f);
                float inv_l = 1.f / l_row;
                if constexpr (FEAT == kDropout) inv_l *= p.drop_inv_keep;   // kept P scaled by 1 / (1 - p)
                // row of O: batch tb (0 when packed) of S rows, then the
                // sequence start `base` (0 unless packed)
                uint16_t* orow = static_cast<uint16_t*>(p.o_ptr) +
                                 ((static_cast<size_t>(ie.tb) * p.S + ie.base + row) * p.H + ie.h) * p.d_head;
                if (eok) {
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int q = 0; q < kDH / 32; ++q) {
                        uint32_t o[32];
                        ptx::tmem_ld_32x32b_x32(tO + q * 32, o);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence<32>(o);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {   // four 16-byte chunks of 8 values
                            const int cc = hf * (kDH / 8) + q * 4 + u;   // chunk along the row
                            uint4 v;
                            v.x = pack2<BF16>(__uint_as_float(o[u * 8 + 0]) * inv_l,
                                              __uint_as_float(o[u * 8 + 1]) * inv_l);
                            v.y = pack2<BF16>(__uint_as_float(o[u * 8 + 2]) * inv_l,
                                              __uint_as_float(o[u * 8 + 3]) * inv_l);
                            v.z = pack2<BF16>(__uint_as_float(o[u * 8 + 4]) * inv_l,
                                              __uint_as_float(o[u * 8 + 5]) * inv_l);
                            v.w = pack2<BF16>(__uint_as_float(o[u * 8 + 6]) * inv_l,
                                              __uint_as_float(o[u * 8 + 7]) * inv_l);
                            if (direct) {
                                if (row < ie.S && cc * 8 < p.d_head) *reinterpret_cast<uint4*>(orow + cc * 8) = v;
                            } else {
                                const int box = cc >> 3;
                                const int phys = (cc & 7) ^ (r & 7);
                                *reinterpret_cast<uint4*>(stage + box * (kBM * 128) + r * 128 + phys * 16) = v;
                            }
                        }
                    }
                    if (!direct) ptx::fence_proxy_async_smem();
                }
                bool all_ok = eok;
                if (!direct) {
                    all_ok = ptx::named_barrier_and(tile_bar, kTileThreads, eok);
                    if (all_ok && store_thread) {
                        for (int cch = 0; cch < kChunks; ++cch)
                            ptx::tma_store_4d(&tmO, ptx::smem_addr(stage + cch * (kBM * 128)), cch * 64, ie.h,
                                              ie.base + r0, ie.tb);
                        ptx::bulk_commit_group();
                    }
                }
                if (kStageInQ && all_ok && store_thread) {
                    // the Q buffer may take the next item's Q once the store has read it
                    if (!direct) ptx::bulk_wait_group_read_all();
                    ptx::mbar_arrive(bar_addr(&bars->q_empty));
                }
                if (eok && hf == 0 && p.lse != nullptr && row < ie.S) {
                    // LSE = scale * m + ln l = ln2 * (m * scale * log2e + log2 l)
                    const size_t li = FEAT == kPacked
                                          ? static_cast<size_t>(ie.h) * p.total + ie.base + row
                                          : static_cast<size_t>(ie.bh) * p.S + row;
                    p.lse[li] = (m_use * c + log2f(l_row)) * 0.69314718055994530942f;
                }
            } else if (kStageInQ && store_thread) {
                // no key tile for this query tile: its Q buffer was never loaded
                release_q();
            }
            gs0 += static_cast<uint32_t>(n_tiles);
            ++ki;
        }
        // every O store must be complete before the CTA exits
        if (store_thread) ptx::bulk_wait_group_all();
        if (FA_DEBUG && store_thread) bars->dbg[5 + t] = static_cast<int>(gs0);
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (FA_DEBUG && threadIdx.x == 0 && !*abort_flag)
        debug_check(bars->dbg[0] == bars->dbg[1] && bars->dbg[1] == bars->dbg[2] &&
                    bars->dbg[3] == bars->dbg[5] && bars->dbg[4] == bars->dbg[6]);
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// Merges the partial results of the split-over-keys path: for each row,
// M = max_s m_s, l = sum_s l_s 2^(m_s - M), O = sum_s o~_s 2^(m_s - M) / l and
// LSE = ln2 (M + log2 l) -- the same rescaling by alpha = exp(m_old - m_new)
// as the online update of section 沿 C fragment 做 Online Softmax, applied
// across splits instead of across tiles.  A CTA covers combine_threads(D) / (D/8) rows of
// one query tile of one (b, h); thread (r, c) produces the 8 outputs of row r,
// columns [8c, 8c+8).  Launched as a programmatic dependent of the main
// kernel: it waits for that grid to complete before reading its partials.
// threads per CTA (measured: 128 is 1-2 % faster than 256 on split shapes
// back to back, with twice the CTAs spread over the SMs; 64 mixed)
#ifndef FA_COMBINE_THREADS
#define FA_COMBINE_THREADS 128
#endif
constexpr int kCombineThreads = FA_COMBINE_THREADS;
constexpr int kCombineMaxSplits = 16;   // weights kept in registers up to this
// threads per CTA for width D: a whole number of rows of D / 8 chunks, and a
// whole number of CTAs per 128-row tile (D = 192: 24 chunks, 8 rows)
__host__ __device__ constexpr int combine_threads(int D) { return D == 192 ? 192 : kCombineThreads; }

template <int D, bool BF16>
__global__ void __launch_bounds__(combine_threads(D)) fa_combine_kernel(const FwdParams p, void* O) {
    constexpr int kCols = D / 8;                        // 8-column chunks per row
    constexpr int kRows = combine_threads(D) / kCols;   // rows per CTA
    constexpr int kPerTile = kBM / kRows;               // CTAs per query tile
    static_assert(combine_threads(D) % kCols == 0 && kBM % kRows == 0, "combine CTA shape");
    const int qt = blockIdx.x / kPerTile;
    const int bh = blockIdx.y;
    const int ns = p.block_splits[qt / kQTiles];
    debug_check(ns >= 1 && ns <= p.max_splits);
    // the next kernel in the stream may start its set-up now (it waits for
    // this grid before touching memory)
    ptx::launch_dependents();
    if (ns <= 1) return;   // this tile was written by the main kernel
    ptx::grid_dependency_wait();
    const int r = (blockIdx.x % kPerTile) * kRows + static_cast<int>(threadIdx.x) % kRows;
    const int cchunk = static_cast<int>(threadIdx.x) / kRows;
    const int row = qt * kBM + r;
    if (row >= p.S) return;
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int ntq = (p.S + kBM - 1) / kBM;
    const size_t slot0 = partial_slot(bh, ntq, qt, p.max_splits, 0);
    const float* ml0 = p.ws_ml + slot0 * (2 * kBM);
    const float4* po0 = reinterpret_cast<const float4*>(p.ws_o + slot0 * static_cast<size_t>(kBM * D));
    constexpr size_t kSlotMl = 2 * kBM;
    constexpr size_t kSlotO = static_cast<size_t>(kBM) * D / 4;   // float4 per slot

    // The loads of every split's (m, l) and o~ chunk are independent of one
    // another: issue them all before any of the arithmetic (one L2 round trip).
    const float4* pa = po0 + (2 * cchunk) * kBM + r;
    float msp[kCombineMaxSplits], lsp[kCombineMaxSplits];
    float4 xo[kCombineMaxSplits], yo[kCombineMaxSplits];
#pragma unroll
    for (int s = 0; s < kCombineMaxSplits; ++s) {
        msp[s] = -INFINITY;
        lsp[s] = 0.f;
        xo[s] = yo[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s < ns) {
            msp[s] = ml0[s * kSlotMl + r];
            lsp[s] = ml0[s * kSlotMl + kBM + r];
            xo[s] = pa[s * kSlotO];
            yo[s] = pa[s * kSlotO + kBM];
        }
    }
    float M = -INFINITY;
    for (int s = kCombineMaxSplits; s < ns; ++s)
        if (ml0[s * kSlotMl + kBM + r] > 0.f) M = fmaxf(M, ml0[s * kSlotMl + r]);
#pragma unroll
    for (int s = 0; s < kCombineMaxSplits; ++s)
        if (lsp[s] > 0.f) M = fmaxf(M, msp[s]);
    float Lsum = 0.f;
#pragma unroll
    for (int s = 0; s < kCombineMaxSplits; ++s) {
        // weight of split s before normalisation (0 when it saw no key)
        msp[s] = lsp[s] > 0.f ? ptx::ex2_approx(msp[s] - M) : 0.f;
        Lsum += lsp[s] * msp[s];
    }
    for (int s = kCombineMaxSplits; s < ns; ++s) {
        const float ls = ml0[s * kSlotMl + kBM + r];
        if (ls > 0.f) Lsum += ls * ptx::ex2_approx(ml0[s * kSlotMl + r] - M);
    }
    const float inv_l = 1.f / Lsum;

    // a split that saw no key wrote no o~ (its chunk is not read into the sum)
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < kCombineMaxSplits; ++s) {
        if (msp[s] > 0.f) {
            const float w = msp[s];
            const float4 x = xo[s], y = yo[s];
            acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
            acc[4] += w * y.x; acc[5] += w * y.y; acc[6] += w * y.z; acc[7] += w * y.w;
        }
    }
    for (int s = kCombineMaxSplits; s < ns; ++s) {
        const float ls = ml0[s * kSlotMl + kBM + r];
        if (!(ls > 0.f)) continue;
        const float w = ptx::ex2_approx(ml0[s * kSlotMl + r] - M);
        const float4 x = pa[s * kSlotO];
        const float4 y = pa[s * kSlotO + kBM];
        acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
        acc[4] += w * y.x; acc[5] += w * y.y; acc[6] += w * y.z; acc[7] += w * y.w;
    }
    uint4 v;
    v.x = pack2<BF16>(acc[0] * inv_l, acc[1] * inv_l);
    v.y = pack2<BF16>(acc[2] * inv_l, acc[3] * inv_l);
    v.z = pack2<BF16>(acc[4] * inv_l, acc[5] * inv_l);
    v.w = pack2<BF16>(acc[6] * inv_l, acc[7] * inv_l);
    uint16_t* out = reinterpret_cast<uint16_t*>(O) +
                    ((static_cast<size_t>(b) * p.S + row) * p.H + h) * p.d_head + cchunk * 8;
    if (cchunk * 8 < p.d_head) *reinterpret_cast<uint4*>(out) = v;
    if (p.lse != nullptr && cchunk == 0)
        p.lse[static_cast<size_t>(bh) * p.S + row] = (M + log2f(Lsum)) * 0.69314718055994530942f;
}

}  // namespace fa

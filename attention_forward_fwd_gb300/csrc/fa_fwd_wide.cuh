// FlashAttention-2 forward for head dimensions 136 .. 256 on sm_103a.
//
// The same computation as fa_fwd_kernel (page "CuTe 详解：以 FlashAttention-2
// 拆解 Layout、TiledCopy 与 TiledMMA": S = Q K^T (section 先看全局), the online
// softmax with the O correction (section 沿 C fragment 做 Online Softmax), the
// second product P V (section V 的转置只发生在视图里) and the O + LSE epilogue
// (section 第二次 GEMM 与输出 Epilogue)), laid out for a wide head of D = 192
// or 256 columns: one 128-row query tile per CTA, so that its S (128 columns)
// and O (D columns) fit in tensor memory: S in two buffers (columns [0, 128)
// and [384, 512)), P written over its S, O in [128, 128 + D).  The tensor
// pipe runs S(0), S(1), P V(0), S(2), P V(1), ...: S(j+1) overlaps the
// softmax of tile j.  S(j) is issued after P V(j-2), so when S(j) is
// complete the P V that last read its buffer is too; O may be rescaled once
// P V(j-1) has reported on its own barrier.
//
// Shared memory holds the Q tile (D / 64 boxes of 64 columns) and two rings:
// K as 128-key x 64-column boxes (16 KiB; S(j) reads box c of K(j) in its
// K steps 4c .. 4c+3 and releases it after them), V as pieces of 128 or 64
// keys x D columns (P V(j) reads a piece in the K steps over its keys).  A
// copy is issued as soon as the slot it goes to is released, several key
// tiles ahead of its use: a copy from L2 under load takes about as long as
// two of the MMAs.  Once the last P V is complete the V ring stages the
// final O tile for its TMA stores.
//
// Warps 0-3: softmax, thread = query row = TMEM lane.  Warp 4: TMEM
// allocation and MMA issue (converged warp, one elected lane).  Warp 5: Q
// and K copies, warp 6: V copies (lane 0 issues; each in the order the MMAs
// release their slots, neither waiting on the other's).  Every wait is
// bounded (wait_phase); after a timeout each role stops, the copy warps wait
// (bounded) for their copies, the MMA warp for its MMAs, and the CTA frees
// its tensor memory and exits.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kWideD = 256;        // the widest head the library takes
constexpr int kWideThreads = 224;  // softmax warps 0-3, MMA warp 4, copy warps 5 (Q, K) and 6 (V)
constexpr int kWideBoxBytes = kBN * 128;   // one 128-key x 64-column box of K
constexpr int kWideMaxKSlots = 6;
constexpr int kWideMaxVSlots = 3;
constexpr uint32_t kWideTmemCols = 512;   // S/P buffers [0, 128) and [384, 512), O [128, 128 + D)
constexpr uint32_t kWideS1 = 384;         // column of the second S/P buffer
// the kernel's width for a head of Dh columns (136 .. 256)
__host__ __device__ constexpr int wide_dim(int Dh) { return Dh <= 192 ? 192 : 256; }
// K and V bytes of the heads whose CTAs are ordered together (a share of the
// 126 MB L2, leaving room for the next group and the Q / O traffic).  Causal
// calls take larger groups: their query tiles differ in cost, and a group
// must hold enough of them for the heaviest-first order to balance the SMs.
constexpr long long kWideL2Share = 16ll << 20;
constexpr long long kWideL2ShareCausal = 32ll << 20;

// The final O tile is staged in shared memory and stored by TMA (1), or
// each softmax thread stores its row from registers (0).
#ifndef FA_WIDE_STAGE_O
#define FA_WIDE_STAGE_O 1
#endif

struct WideBars {
    uint64_t q_full;
    uint64_t kbox_full[kWideMaxKSlots];    // K slot holds its box
    uint64_t kbox_empty[kWideMaxKSlots];   // ... and S has read it
    uint64_t v_full[kWideMaxVSlots];       // V slot holds its piece
    uint64_t v_empty[kWideMaxVSlots];      // ... and P V has read it
    uint64_t s_full[2];     // S(j) complete in buffer j % 2 (and every MMA before it)
    // P(j) stored in buffer j % 2 by the 128 softmax threads.  One barrier
    // per buffer: S(j+1) is issued before the MMA warp waits for P(j), so the
    // softmax may store P(j+1) before that wait is seen, and a single barrier
    // could move two phases past it; P(j+2) needs S(j+2), which is issued
    // only after P V(j)
    uint64_t p_full[2];
    uint64_t o_done;        // one phase per P V(j)
    // the last P V complete: the epilogue cannot wait on o_done, which may
    // then be one, two or no phases short of it (parity tells two apart)
    uint64_t o_last;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

template <int D>
struct WideSmem {
    static_assert(D == 192 || D == 256, "wide head widths");
    static_assert(kBN + D <= static_cast<int>(kWideS1), "O overlaps the second S/P buffer");
    static constexpr int kAtoms = D / 64;              // 64-column boxes per row
    static constexpr int kTileBytes = kBM * D * 2;     // one 128 x D 16-bit tile
    // K ring: kKSlots boxes.  V ring: kVSlots pieces, each kVRows keys of a
    // tile (a V tile in kVSplit pieces).  Sized to fill the 227 KiB.
    static constexpr int kKSlots = D == 192 ? 5 : 4;
    static constexpr int kVSplit = D == 192 ? 1 : 2;
    static constexpr int kVSlots = D == 192 ? 2 : 3;
    static constexpr int kVRows = kBN / kVSplit;
    static constexpr int kVBoxBytes = kVRows * 128;    // one 64-column box of a piece
    static constexpr int kVPieceBytes = kAtoms * kVBoxBytes;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kTileBytes;
    static constexpr int kOffV = kOffK + kKSlots * kWideBoxBytes;
    static constexpr int kOffBar = kOffV + kVSlots * kVPieceBytes;
    static constexpr int kAlloc = kOffBar + static_cast<int>(sizeof(WideBars)) + 1024;
    static_assert(kKSlots >= kAtoms && kKSlots <= kWideMaxKSlots, "K ring");
    static_assert(kVSlots >= kVSplit && kVSlots <= kWideMaxVSlots && kVRows % 64 == 0, "V ring");
    static_assert(kAlloc <= 232448, "shared memory beyond the 227 KiB a CTA may use");
};

// Work item x of the grid.  Heads are taken in groups whose K and V fit in
// kWideL2Share (causal: kWideL2ShareCausal) bytes together; inside a group,
// heads fastest and query tiles heaviest first when causal.  The CTAs of a
// group run at about the same
// time, so each head's K / V comes from DRAM about once, where an order over
// all heads at once read every head's prefix again in every wave of CTAs.
// DROP: attention dropout (the draws of fa_fwd_kernel's dropout variant:
// Philox4x32-10 blocks with counter (key / 8, row, head, batch) and the seed
// as key, sixteen-bit draws; kept P scaled by 1 / (1 - p) in the epilogue).
template <int D, bool BF16, bool DROP>
__global__ void __launch_bounds__(kWideThreads, 1)
    fa_fwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                       const FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    using L = WideSmem<D>;
    constexpr int kAtoms = L::kAtoms;
    constexpr int kTileBytes = L::kTileBytes;
    WideBars* bars = reinterpret_cast<WideBars*>(smem + L::kOffBar);
    volatile int* abort_flag = &bars->abort;
    auto bar = [&](const uint64_t* b) { return ptx::smem_addr(b); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ------------------------------------------------------------ the item
    const int bhn = p.B * p.H;
    const int ntq = (p.S + kBM - 1) / kBM;
    const bool causal = p.causal != 0;
    // K and V bytes (16-bit) per query head: query heads h .. h + kv_group - 1
    // share one K/V head, so a group of them holds 1/kv_group of that each
    const long long kv_head_bytes = max(1ll, 4ll * p.S * p.d_head / p.kv_group);
    const int group = static_cast<int>(max(
        1ll, min(static_cast<long long>(bhn), (causal ? kWideL2ShareCausal : kWideL2Share) / kv_head_bytes)));
    // split over keys (kv_chunk > 0): CTA blockIdx.x runs split s = blockIdx.x
    // % max_splits of query tile x = blockIdx.x / max_splits, the key tiles
    // [s * kv_chunk, (s + 1) * kv_chunk) of its range (possibly none)
    const int nsplit = p.kv_chunk > 0 ? p.max_splits : 1;
    const int x = static_cast<int>(blockIdx.x) / nsplit;
    const int split = static_cast<int>(blockIdx.x) - x * nsplit;
    const int g0 = (x / (group * ntq)) * group;   // first head of x's group
    const int gsize = min(group, bhn - g0);
    const int local = x - g0 * ntq;               // in [0, gsize * ntq)
    const int y = local / gsize;
    const int bh = g0 + (local - y * gsize);
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int hkv = h / p.kv_group;
    const int qt = causal ? (ntq - 1 - y) : y;
    const int r0 = qt * kBM;
    // The item's sequence: S_b rows from row `base` of batch `tb` of the
    // tensors.  Packed batches (cu_seqlens) are one batch of `total` rows,
    // sequence b rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (at most S); their
    // offsets are read after the previous kernel in the stream has finished.
    int S_b = p.S, base = 0, tb = b;
    if (p.cu_seqlens != nullptr) {
        ptx::grid_dependency_wait();
        const int a = p.cu_seqlens[b];
        const int e = p.cu_seqlens[b + 1];
        const bool bad = !(a >= 0 && e >= a && e <= p.total && e - a <= p.S);
        if (bad && qt == 0 && h == 0 && split == 0 && threadIdx.x == 0)
            atomicCAS(&g_fa_device_status, 0, kStatusBadSeqlens);
        S_b = bad ? 0 : e - a;
        base = bad ? 0 : a;
        tb = 0;
    }
    // key tiles [lo, hi) that the tile's rows see: up to the diagonal when
    // causal, and within [row - win_left, row + win_right] for a local window
    int lo = 0, hi = key_tiles_for(r0, S_b, causal);   // 0 past the sequence's end
    if (p.win_left >= 0) lo = min(hi, max(0, r0 - p.win_left) / kBN);
    if (p.win_right >= 0) hi = min(hi, (r0 + kBM - 1 + p.win_right) / kBN + 1);
    const int n_all = max(0, hi - lo);
    const int jb = lo + split * p.kv_chunk;             // first key tile of this CTA
    const int n_tiles = p.kv_chunk > 0 ? max(0, min(hi, jb + p.kv_chunk) - jb) : n_all;
    debug_check(qt >= 0 && qt < ntq && bh < bhn && (n_all >= 1 || r0 >= S_b) && split < nsplit &&
                (p.kv_chunk == 0 || (p.cu_seqlens == nullptr && p.win_left < 0 && p.win_right < 0)));

    if (threadIdx.x == 32 * 5) {
        ptx::mbar_init(bar(&bars->q_full), 1);
        for (int s = 0; s < L::kKSlots; ++s) {
            ptx::mbar_init(bar(&bars->kbox_full[s]), 1);
            ptx::mbar_init(bar(&bars->kbox_empty[s]), 1);
        }
        for (int s = 0; s < L::kVSlots; ++s) {
            ptx::mbar_init(bar(&bars->v_full[s]), 1);
            ptx::mbar_init(bar(&bars->v_empty[s]), 1);
        }
        ptx::mbar_init(bar(&bars->s_full[0]), 1);
        ptx::mbar_init(bar(&bars->s_full[1]), 1);
        ptx::mbar_init(bar(&bars->p_full[0]), kBM);
        ptx::mbar_init(bar(&bars->p_full[1]), kBM);
        ptx::mbar_init(bar(&bars->o_done), 1);
        ptx::mbar_init(bar(&bars->o_last), 1);
        ptx::mbar_init(bar(&bars->drain), 1);
        bars->abort = 0;
        ptx::fence_barrier_init();
        ptx::tma_prefetch_map(&tmQ);
        ptx::tma_prefetch_map(&tmK);
        ptx::tma_prefetch_map(&tmV);
        ptx::tma_prefetch_map(&tmO);
    }
    if (warp == 4) {
        ptx::tmem_alloc(ptx::smem_addr(&bars->tmem_base), kWideTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    ptx::launch_dependents();

    auto wait_warp = [&](uint32_t b_, uint32_t parity, bool honour_abort = true) {
        return __all_sync(0xffffffffu, wait_phase(b_, parity, abort_flag, honour_abort));
    };

    if (warp == 5) {
        // ---------------------------------------------------- Q and K copies
        ptx::grid_dependency_wait();   // the previous kernel may write Q, K, V
        const bool q_issued = n_tiles > 0 && !p.drop_first_q;
        if (lane == 0 && q_issued) {
            const uint32_t full = bar(&bars->q_full);
            ptx::mbar_arrive_expect_tx(full, kTileBytes);
            for (int c = 0; c < kAtoms; ++c)
                ptx::tma_load_4d(sbase + L::kOffQ + c * (kBM * 128), &tmQ, full, c * 64, h, base + r0, tb);
        }
        // box n = i * kAtoms + c (box c of K(i)) goes to slot n % kKSlots as
        // its (n / kKSlots)-th box, once S has read the slot's previous one
        const uint32_t k0 = sbase + L::kOffK;
        const int nbox = n_tiles * kAtoms;
        int n = 0;
        for (; n < nbox; ++n) {
            const int slot = n % L::kKSlots;
            const int use = n / L::kKSlots;
            if (use > 0 && !wait_warp(bar(&bars->kbox_empty[slot]), static_cast<uint32_t>((use - 1) & 1))) break;
            if (lane == 0) {
                const int i = n / kAtoms;
                const int c = n - i * kAtoms;
                const uint32_t full = bar(&bars->kbox_full[slot]);
                ptx::mbar_arrive_expect_tx(full, kWideBoxBytes);
                ptx::tma_load_4d(k0 + slot * kWideBoxBytes, &tmK, full, c * 64, hkv, base + (jb + i) * kBN, tb);
            }
        }
        if (*abort_flag) {
            // let every copy this warp started land before the CTA exits
            // (only the last box of each slot can still be in flight)
            if (q_issued) wait_warp(bar(&bars->q_full), 0, false);
            for (int m = max(0, n - L::kKSlots); m < n; ++m)
                wait_warp(bar(&bars->kbox_full[m % L::kKSlots]), static_cast<uint32_t>((m / L::kKSlots) & 1), false);
        }
    } else if (warp == 6) {
        // ---------------------------------------------------------- V copies
        ptx::grid_dependency_wait();
        // V(0) is first read after S(0), S(1) and the softmax of tile 0:
        // its copies wait for Q, whose copy and K(0)'s they would slow
        bool ok = n_tiles == 0 || wait_warp(bar(&bars->q_full), 0);
        // piece m = i * kVSplit + e (keys [e * kVRows, (e + 1) * kVRows) of
        // V(i)) goes to slot m % kVSlots, once P V has read the slot's
        // previous piece
        const uint32_t v0 = sbase + L::kOffV;
        const int npiece = n_tiles * L::kVSplit;
        int m = 0;
        for (; m < npiece && ok; ++m) {
            const int slot = m % L::kVSlots;
            const int use = m / L::kVSlots;
            if (use > 0 && !(ok = wait_warp(bar(&bars->v_empty[slot]), static_cast<uint32_t>((use - 1) & 1)))) break;
            if (lane == 0) {
                const int i = m / L::kVSplit;
                const int e = m - i * L::kVSplit;
                const uint32_t full = bar(&bars->v_full[slot]);
                ptx::mbar_arrive_expect_tx(full, L::kVPieceBytes);
                for (int c = 0; c < kAtoms; ++c)
                    ptx::tma_load_4d(v0 + slot * L::kVPieceBytes + c * L::kVBoxBytes, &tmV, full, c * 64, hkv,
                                     base + (jb + i) * kBN + e * L::kVRows, tb);
            }
        }
        if (*abort_flag)
            for (int q = max(0, m - L::kVSlots); q < m; ++q)
                wait_warp(bar(&bars->v_full[q % L::kVSlots]), static_cast<uint32_t>((q / L::kVSlots) & 1), false);
    } else if (warp == 4) {
        // ------------------------------------------------------ MMA issue
        constexpr uint32_t kIdescQK = ptx::idesc_f16_f32(kBM, kBN, BF16, false);
        constexpr uint32_t kIdescPV = ptx::idesc_f16_f32(kBM, D, BF16, true);
        const uint32_t hi = ptx::sdesc_sw128_hi(1024);
        const uint32_t qlo = ptx::sdesc_sw128_lo(sbase + L::kOffQ, 16);
        const uint32_t klo = ptx::sdesc_sw128_lo(sbase + L::kOffK, 16);
        // V MN-major (rows are keys): the 64-column boxes of a piece
        // kVBoxBytes apart
        const uint32_t vlo = ptx::sdesc_sw128_lo(sbase + L::kOffV, L::kVBoxBytes);
        bool ok = n_tiles == 0 || wait_warp(bar(&bars->q_full), 0);
        // S(i) into buffer i % 2: Q K(i)^T over the D columns, box by box
        // (four K=16 steps of 32 bytes inside a box), each box handed back
        // to the K ring once its steps have run
        auto issue_s = [&](int i) {
            const uint32_t d = tmem + ((i & 1) ? kWideS1 : 0u);
#pragma unroll
            for (int c = 0; c < kAtoms; ++c) {
                const int n = i * kAtoms + c;
                const int slot = n % L::kKSlots;
                if (!(ok = wait_warp(bar(&bars->kbox_full[slot]), static_cast<uint32_t>((n / L::kKSlots) & 1))))
                    return;
                ptx::tc_fence_after_sync();
                ptx::mma_ss_x4_lo(d, qlo + c * (kBM * 128 / 16), klo + slot * (kWideBoxBytes / 16), hi, 2u, kIdescQK,
                                  c > 0 ? 1u : 0u);
                ptx::tc_commit_warp(bar(&bars->kbox_empty[slot]));
            }
            ptx::tc_commit_warp(bar(&bars->s_full[i & 1]));
        };
        if (ok && n_tiles > 0) issue_s(0);
        for (int j = 0; j < n_tiles && ok; ++j) {
            if (j + 1 < n_tiles) {
                issue_s(j + 1);
                if (!ok) break;
            }
            // O (+)= P(j) V(j): P from the first 64 columns of S(j)'s buffer
            // (8 columns per K step of 16 keys), V piece by piece
            if (!(ok = wait_warp(bar(&bars->p_full[j & 1]), static_cast<uint32_t>((j >> 1) & 1)))) break;
            const uint32_t pa = tmem + ((j & 1) ? kWideS1 : 0u);
#pragma unroll
            for (int e = 0; e < L::kVSplit; ++e) {
                const int m = j * L::kVSplit + e;
                const int slot = m % L::kVSlots;
                if (!(ok = wait_warp(bar(&bars->v_full[slot]), static_cast<uint32_t>((m / L::kVSlots) & 1)))) break;
                ptx::tc_fence_after_sync();
                const uint32_t vs = vlo + slot * (L::kVPieceBytes / 16);
#pragma unroll
                for (int kk = 0; kk < L::kVRows / 16; kk += 4) {
                    const int kg = e * (L::kVRows / 16) + kk;   // K step within the tile
                    ptx::mma_ts_x4_lo(tmem + kBN, pa + kg * 8, vs + kk * (16 * 128 / 16), hi, 8u, 16u * 128u / 16u,
                                      kIdescPV, (j > 0 || kg > 0) ? 1u : 0u);
                }
                ptx::tc_commit_warp(bar(&bars->v_empty[slot]));
            }
            if (!ok) break;
            ptx::tc_commit_warp(bar(&bars->o_done));
            if (j + 1 == n_tiles) ptx::tc_commit_warp(bar(&bars->o_last));
        }
        // every MMA must be complete before the tensor memory is freed
        ptx::tc_commit_warp(bar(&bars->drain));
        wait_warp(bar(&bars->drain), 0, false);
    } else {
        // --------------------------------------------------------- softmax
        const int r = static_cast<int>(threadIdx.x);   // row of the tile, TMEM lane
        const int row = r0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
        const uint32_t tS0 = tmem + lane_off;            // S(j), then P(j) over it, buffer j % 2
        const uint32_t tO = tmem + lane_off + kBN;       // O, D columns
        const float c = p.scale_log2;
        float m_use = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            ok = ok && wait_phase(bar(&bars->s_full[j & 1]), static_cast<uint32_t>((j >> 1) & 1), abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after_sync();
            const uint32_t tS = tS0 + ((j & 1) ? kWideS1 : 0u);
            uint32_t s[kBN];
#pragma unroll
            for (int q = 0; q < kBN / 32; ++q) ptx::tmem_ld_32x32b_x32(tS + q * 32, s + q * 32);
            ptx::tmem_ld_wait();
            ptx::reg_fence<kBN>(s);
            // keys outside [first, last] are masked: past the sequence, after
            // the row (causal) or outside the window
            const int kv0 = (jb + j) * kBN;
            int last = causal ? min(S_b - 1, row) : (S_b - 1);
            if (p.win_right >= 0) last = min(last, row + p.win_right);
            const int first = p.win_left >= 0 ? row - p.win_left : -1;
            if (kv0 + kBN - 1 > last || kv0 < first) {
#pragma unroll
                for (int kq = 0; kq < kBN; ++kq)
                    if (kv0 + kq > last || kv0 + kq < first) s[kq] = __float_as_uint(-INFINITY);
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int kq = 0; kq < kBN / 2; ++kq)
                mx[kq % 4] = ptx::fmax3(mx[kq % 4], __uint_as_float(s[2 * kq]), __uint_as_float(s[2 * kq + 1]));
            const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            const float m_new = fmaxf(m_use, m_tile);
            // lazy rescale: move the reference only when the max grew by more
            // than kTauLog2 (log2 units); the first tile always moves it
            float alpha = 1.f;
            const bool rescale = (m_new - m_use) * c > kTauLog2;
            if (rescale) {
                alpha = ptx::ex2_approx((m_use - m_new) * c);   // 0 on the first tile
                m_use = m_new;
            }
            // rows whose reference moved scale O by alpha, once P V(j-1) is
            // complete (phase j-1 of o_done: P V(j-2) is complete already, as
            // S(j) was issued after it, and P V(j) waits for this P(j))
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                ok = wait_phase(bar(&bars->o_done), static_cast<uint32_t>((j - 1) & 1), abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ptx::tc_fence_after_sync();
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    ptx::tmem_ld_32x32b_x32(tO + q * 32, o);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence<32>(o);
#pragma unroll
                    for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
                    ptx::tmem_st_32x32b_x32(tO + q * 32, o);
                }
            }
            // (a row whose keys so far all lie outside its window has no
            // reference yet: its p are 0)
            const float mc = (m_use == -INFINITY) ? 0.f : m_use * c;
            const float2 c2 = make_float2(c, c);
            const float2 nmc2 = make_float2(-mc, -mc);
            float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int q = 0; q < kBN / 32; ++q) {
                uint32_t pk[16];
                uint32_t dw[16] = {};   // dropout draws of these 32 keys (two per word)
                if constexpr (DROP)
                    philox4x32_10<4>(static_cast<uint32_t>(kv0 + q * 32) >> 3, static_cast<uint32_t>(row),
                                     static_cast<uint32_t>(h), static_cast<uint32_t>(b), p.drop_seed_lo,
                                     p.drop_seed_hi, dw);
#pragma unroll
                for (int kq = 0; kq < 16; ++kq) {
                    const float2 xv = __ffma2_rn(make_float2(__uint_as_float(s[q * 32 + 2 * kq]),
                                                             __uint_as_float(s[q * 32 + 2 * kq + 1])),
                                                 c2, nmc2);
                    const float2 pp = make_float2(ptx::ex2_approx(xv.x), ptx::ex2_approx(xv.y));
                    sum2[kq & 1] = __fadd2_rn(sum2[kq & 1], pp);
                    pk[kq] = pack_p<DROP ? kDropout : kPlain, BF16>(p, pp, dw[kq]);
                }
                ptx::tmem_st_32x32b_x16(tS + q * 16, pk);
            }
            const float2 sum = __fadd2_rn(sum2[0], sum2[1]);
            l = l * alpha + (sum.x + sum.y);
            ptx::tmem_st_wait();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar(&bars->p_full[j & 1]));
        }
        // ---------------------------------------------------------- epilogue
        ok = ok && (n_tiles == 0 || wait_phase(bar(&bars->o_last), 0, abort_flag));
        ok = __all_sync(0xffffffffu, ok);
        if (p.kv_chunk > 0) {
            // partial result of this split (the layout of fa_fwd_kernel's split
            // path: o~ as [D/4][128] float4, then m (log2 units) and l per
            // row); a split with no key records l = 0 and m = -inf
            const size_t slot = partial_slot(bh, ntq, qt, p.max_splits, split);
            float* ml = p.ws_ml + slot * (2 * kBM);
            float4* po = reinterpret_cast<float4*>(p.ws_o + slot * static_cast<size_t>(kBM * D));
            if (ok && n_tiles > 0) {
                ptx::tc_fence_after_sync();
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    ptx::tmem_ld_32x32b_x32(tO + q * 32, o);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence<32>(o);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        po[(q * 8 + u) * kBM + r] = make_float4(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1]),
                                                                __uint_as_float(o[4 * u + 2]), __uint_as_float(o[4 * u + 3]));
                }
                ml[r] = m_use * c;
                ml[kBM + r] = l;
            } else if (ok) {
                ml[r] = -INFINITY;
                ml[kBM + r] = 0.f;
            }
        } else if (n_tiles > 0) {
            // final result: staged as the 128-byte-swizzled TMA boxes in the
            // V ring (every P V is complete, so nothing reads it any more),
            // each box stored by one thread once all rows have written it;
            // rows past S are dropped by the store.  The last tile of a packed sequence is stored row by row
            // instead (the rows after it belong to the next sequence).
            const bool direct = FA_WIDE_STAGE_O == 0 || (p.cu_seqlens != nullptr && r0 + kBM > S_b);
            uint8_t* stage = smem + L::kOffV;
            float inv_l = 1.f / l;
            if constexpr (DROP) inv_l *= p.drop_inv_keep;   // kept P scaled by 1 / (1 - p)
            // row of O: batch tb (0 when packed) of S rows, then the sequence
            // start `base` (0 unless packed)
            uint16_t* orow = static_cast<uint16_t*>(p.o_ptr) +
                             ((static_cast<size_t>(tb) * p.S + base + row) * p.H + h) * p.d_head;
            // eight values of O's row, scaled and rounded to 16 bits
            auto pack8 = [&](const uint32_t* o) {
                uint4 v;
                v.x = pack2<BF16>(__uint_as_float(o[0]) * inv_l, __uint_as_float(o[1]) * inv_l);
                v.y = pack2<BF16>(__uint_as_float(o[2]) * inv_l, __uint_as_float(o[3]) * inv_l);
                v.z = pack2<BF16>(__uint_as_float(o[4]) * inv_l, __uint_as_float(o[5]) * inv_l);
                v.w = pack2<BF16>(__uint_as_float(o[6]) * inv_l, __uint_as_float(o[7]) * inv_l);
                return v;
            };
            if (!direct) {
                // box by box (64 columns per TMEM round trip): box c is
                // stored while box c + 1 is staged
                if (ptx::named_barrier_and(1, kBM, ok)) {
                    ptx::tc_fence_after_sync();
#pragma unroll 1
                    for (int cb = 0; cb < kAtoms; ++cb) {
                        uint32_t o[64];
                        ptx::tmem_ld_32x32b_x32(tO + cb * 64, o);
                        ptx::tmem_ld_32x32b_x32(tO + cb * 64 + 32, o + 32);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence<64>(o);
                        uint8_t* box = stage + cb * (kBM * 128) + r * 128;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            *reinterpret_cast<uint4*>(box + ((u ^ (r & 7)) * 16)) = pack8(o + u * 8);
                        ptx::fence_proxy_async_smem();
                        ptx::named_barrier_sync(1, kBM);
                        if (threadIdx.x == 0) {
                            ptx::tma_store_4d(&tmO, ptx::smem_addr(stage + cb * (kBM * 128)), cb * 64, h, base + r0, tb);
                            ptx::bulk_commit_group();
                        }
                    }
                    // the CTA's shared memory must outlive the stores' reads
                    if (threadIdx.x == 0) ptx::bulk_wait_group_read_all();
                }
            } else if (ok) {
                ptx::tc_fence_after_sync();
#pragma unroll 1
                for (int q = 0; q < D / 32; q += 2) {
                    uint32_t o[64];
                    ptx::tmem_ld_32x32b_x32(tO + q * 32, o);
                    ptx::tmem_ld_32x32b_x32(tO + q * 32 + 32, o + 32);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence<64>(o);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int col = q * 32 + u * 8;
                        if (row < S_b && col < p.d_head) *reinterpret_cast<uint4*>(orow + col) = pack8(o + u * 8);
                    }
                }
            }
            if (ok && p.lse != nullptr && row < S_b) {
                const size_t li = p.cu_seqlens != nullptr ? static_cast<size_t>(h) * p.total + base + row
                                                          : static_cast<size_t>(bh) * p.S + row;
                p.lse[li] = (m_use * c + log2f(l)) * 0.69314718055994530942f;
            }
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 4) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kWideTmemCols);
    }
}

}  // namespace fa

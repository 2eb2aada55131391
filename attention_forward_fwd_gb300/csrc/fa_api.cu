// fa_api.cu -- C-ABI entry points of libfa_gb300.so (declared in
// include/fa_gb300.h): argument validation, TMA tensor maps, kernel choice
// and launch.  No device memory is allocated and nothing is synchronised.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "fa_fwd_kernel.cuh"
#include "fa_fwd_wide.cuh"
#include "fa_gb300.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, resolved through the runtime so that the
// library does not link against libcuda.
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [B, S, H, D] 16-bit tensor seen as 4-D (D, H, S, B), innermost first; the
// box is 64 elements of D (128 bytes, the 128-byte swizzle span) x 1 head x
// `rows` positions x 1 batch.  Positions past S read as zero and are not
// written by stores.
bool make_map(CUtensorMap* m, const void* base, bool bf16, int B, int S, int H, int D, int rows) {
    EncodeTiledFn enc = encode_tiled();
    if (enc == nullptr) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(H) * D * 2,
                                   static_cast<cuuint64_t>(S) * H * D * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r =
        enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// softmax threads per query row, per head dimension
#ifndef FA_ROW_SPLIT_D64
#define FA_ROW_SPLIT_D64 1
#endif
#ifndef FA_ROW_SPLIT_D128
#define FA_ROW_SPLIT_D128 2
#endif
constexpr int kRowSplitD64 = FA_ROW_SPLIT_D64;
constexpr int kRowSplitD128 = FA_ROW_SPLIT_D128;
// K / V ring slots per head dimension
#ifndef FA_RING_D64
#define FA_RING_D64 6
#endif
#ifndef FA_RING_D128
#define FA_RING_D128 4
#endif
constexpr int kRingD64 = FA_RING_D64;
constexpr int kRingD128 = FA_RING_D128;

// SMs of the current device (0 if it cannot be read), looked up once per
// device; host threads may call concurrently.
int num_sms() {
    static std::once_flag once[64];
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::call_once(once[dev], [&] {
        int n = 0;
        cached[dev] = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? n : 0;
    });
    return cached[dev];
}

// The kernel's parameters (four tensor maps and FwdParams) must fit the 4 KiB
// of a launch's parameter space.
static_assert(sizeof(fa::FwdParams) + 4 * sizeof(CUtensorMap) <= 4096, "kernel parameters too large");
// the device status word carries the host's codes
static_assert(fa::kStatusTimeout == FA_ERR_TIMEOUT && fa::kStatusBadSeqlens == FA_ERR_BAD_SEQLENS &&
                  fa::kStatusDeviceCheck == FA_ERR_DEVICE_CHECK,
              "device status codes");

// Head dimensions the library takes: multiples of 8 up to 256 (the row
// strides of the tensor maps must be multiples of 16 bytes).  D = 64, 128,
// 192 and 256 run at full width; any other runs on the next kernel up, whose
// extra columns the tensor maps read as zeros.  D > 128 has a kernel of its
// own (fa_fwd_wide_kernel, one query tile per CTA, at width 192 or 256).
bool supported_dim(int D) { return D >= 8 && D <= fa::kWideD && D % 8 == 0; }
int kernel_dim(int D) { return D <= 64 ? 64 : D <= 128 ? 128 : fa::wide_dim(D); }

// Cost model of the multi-wave split plans (plan_split_uncached), in key
// steps: an item's cost beyond its key tiles, and the merge's.
#ifndef FA_PLAN_ITEM_D64
#define FA_PLAN_ITEM_D64 1.5
#endif
#ifndef FA_PLAN_MERGE_D64
#define FA_PLAN_MERGE_D64 3.0
#endif
#ifndef FA_PLAN_ITEM_D128
#define FA_PLAN_ITEM_D128 1.0
#endif
#ifndef FA_PLAN_MERGE_D128
#define FA_PLAN_MERGE_D128 1.5
#endif

// How the keys of each query block are split over CTAs: the splits of every
// query block and the work items of one head in the order the kernel visits
// them (the same for every head).
struct SplitPlan {
    int chunk = 0;          // nonzero: split mode
    int max_splits = 1;     // splits of the most split query block
    int ctas_per_head = 0;  // work items per head
    uint8_t ns[fa::kMaxSplitBlocks] = {};       // splits of each query block
    uint32_t item[fa::kMaxSplitItems] = {};     // (block, split, splits) per item
};

SplitPlan no_split(int S) {
    SplitPlan plan;
    plan.ctas_per_head = (S + fa::kQTiles * fa::kBM - 1) / (fa::kQTiles * fa::kBM);
    std::fill(plan.ns, plan.ns + fa::kMaxSplitBlocks, uint8_t{1});
    return plan;
}

long long ctas_per_head_for(int S, bool causal, int chunk) {
    const int nqb = (S + fa::kQTiles * fa::kBM - 1) / (fa::kQTiles * fa::kBM);
    long long n = 0;
    for (int qb = 0; qb < nqb; ++qb) n += (fa::key_tiles_for_block(qb, S, causal) + chunk - 1) / chunk;
    return n;
}

// Fills the item list of a plan from its per-block splits: items longest
// first (each split's key tiles), the splits of a block together, ties in
// the unsplit order (heaviest query block first when causal).  Returns false
// if the head has too many items for the kernel's table.
bool order_items(SplitPlan& plan, int S, bool causal) {
    const int nqb = (S + fa::kQTiles * fa::kBM - 1) / (fa::kQTiles * fa::kBM);
    struct Piece { int len, visit, qb, split, n; };
    Piece pieces[fa::kMaxSplitItems];
    int np = 0;
    plan.max_splits = 1;
    for (int v = 0; v < nqb; ++v) {
        const int qb = causal ? nqb - 1 - v : v;
        const int T = fa::key_tiles_for_block(qb, S, causal);
        const int n = std::max(1, static_cast<int>(plan.ns[qb]));
        const int c = (T + n - 1) / n;
        plan.max_splits = std::max(plan.max_splits, n);
        for (int sp = 0; sp < n; ++sp) {
            if (np == fa::kMaxSplitItems) return false;
            pieces[np++] = Piece{std::min(T, (sp + 1) * c) - sp * c, v, qb, sp, n};
        }
    }
    std::stable_sort(pieces, pieces + np, [](const Piece& a, const Piece& b) { return a.len > b.len; });
    for (int y = 0; y < np; ++y)
        plan.item[y] = static_cast<uint32_t>(pieces[y].qb) | (static_cast<uint32_t>(pieces[y].split) << 8) |
                       (static_cast<uint32_t>(pieces[y].n) << 20);
    plan.ctas_per_head = np;
    return true;
}

// Makespan, in key-tile steps, of the kernel's static schedule (item w of
// round k goes to CTA w mod G, every other round in reverse; items are
// numbered y * BH + bh) when every item costs its key tiles plus `per_item`,
// plus `merge` when some block is split.
double simulate_plan(const SplitPlan& plan, int S, bool causal, long long bh, int sms, double per_item,
                     double merge) {
    int len[fa::kMaxSplitItems];
    bool split = false;
    for (int y = 0; y < plan.ctas_per_head; ++y) {
        const uint32_t e = plan.item[y];
        const int qb = static_cast<int>(e & 0xffu), sp = static_cast<int>((e >> 8) & 0xfffu);
        const int n = std::max(1, static_cast<int>(e >> 20));
        const int T = fa::key_tiles_for_block(qb, S, causal);
        const int c = (T + n - 1) / n;
        len[y] = std::min(T, (sp + 1) * c) - sp * c;
        split = split || n > 1;
    }
    const long long items = bh * plan.ctas_per_head;
    const long long G = std::min<long long>(items, sms);
    std::vector<double> load(static_cast<size_t>(G), 0.0);
    long long c = 0, k = 0;   // item w = y * bh + i goes to round k = w / G, slot c = w % G
    for (int y = 0; y < plan.ctas_per_head; ++y) {
        const double cost = len[y] + per_item;
        for (long long i = 0; i < bh; ++i) {
            load[static_cast<size_t>((k & 1) ? G - 1 - c : c)] += cost;
            if (++c == G) {
                c = 0;
                ++k;
            }
        }
    }
    return *std::max_element(load.begin(), load.end()) + (split ? merge : 0.0);
}

// Split the keys only when one CTA per query block leaves SMs idle:
// * less than three quarters of a wave: the smallest uniform chunk (>= 2
//   key tiles) whose grid still fits in one wave of `sms` CTAs;
// * one to four waves with a ragged last one: the per-block splits whose
//   simulated schedule (simulate_plan) is shortest, if it beats the unsplit
//   schedule by 8 % or more.  Candidates split every block above a key-tile
//   cap, or the m lightest or heaviest blocks into 2-4 pieces (m on a grid
//   of at most ~16 values; only with `multiwave`).  Planned once per shape
//   (cached below): at most ~2 ms of host time for the largest shapes.
// The wide kernel (D > 128, one CTA per 128-row query tile): when the
// tiles fill less than three quarters of a wave, every tile's keys are
// divided into the same number of chunks (at most the merge kernel's
// register-held splits), so that the CTAs come close to one per SM.
SplitPlan plan_split_wide(int B, int H, int S, int sms) {
    SplitPlan plan = no_split(S);
    const long long tiles = static_cast<long long>(B) * H * ((S + fa::kBM - 1) / fa::kBM);
    const int max_kt = (S + fa::kBN - 1) / fa::kBN;
    const int nqb = (S + fa::kQTiles * fa::kBM - 1) / (fa::kQTiles * fa::kBM);
    if (sms <= 0 || tiles * 4 >= static_cast<long long>(sms) * 3 || max_kt < 2 || nqb > fa::kMaxSplitBlocks)
        return plan;
    int ns = static_cast<int>(std::min<long long>(std::min<long long>(fa::kCombineMaxSplits, max_kt), sms / tiles));
    if (ns < 2) return plan;
    const int chunk = (max_kt + ns - 1) / ns;
    ns = (max_kt + chunk - 1) / chunk;
    if (ns < 2) return plan;
    plan.chunk = chunk;
    plan.max_splits = ns;
    plan.ctas_per_head = ((S + fa::kBM - 1) / fa::kBM) * ns;
    std::fill(plan.ns, plan.ns + nqb, static_cast<uint8_t>(ns));
    return plan;
}

SplitPlan plan_split_uncached(int B, int H, int S, int D, bool causal, int sms, bool multiwave) {
    if (kernel_dim(D) > 128) return plan_split_wide(B, H, S, sms);
    SplitPlan plan = no_split(S);
    if (sms <= 0) return plan;
    const int rows_per_cta = fa::kQTiles * fa::kBM;
    const int nqb = (S + rows_per_cta - 1) / rows_per_cta;
    const int nkv_all = (S + fa::kBN - 1) / fa::kBN;
    const long long bh = static_cast<long long>(B) * H;
    const long long base = bh * nqb;
    if (nkv_all <= 2 || nqb > fa::kMaxSplitBlocks) return plan;
    int T[fa::kMaxSplitBlocks];
    for (int qb = 0; qb < nqb; ++qb) T[qb] = fa::key_tiles_for_block(qb, S, causal);
    auto with_splits = [&](auto ns_of) {
        SplitPlan cand;
        cand.chunk = 1;
        for (int qb = 0; qb < nqb; ++qb)
            cand.ns[qb] = static_cast<uint8_t>(std::max(1, std::min({ns_of(qb), T[qb], 255})));
        if (!order_items(cand, S, causal)) cand.chunk = 0;
        return cand;
    };
    if (base * 4 < static_cast<long long>(sms) * 3) {
        int lo = 2, hi = nkv_all;   // grid size is non-increasing in the chunk
        if (bh * ctas_per_head_for(S, causal, hi) > sms) return plan;
        while (lo < hi) {
            const int mid = (lo + hi) / 2;
            if (bh * ctas_per_head_for(S, causal, mid) <= sms) hi = mid;
            else lo = mid + 1;
        }
        if ((nkv_all + lo - 1) / lo <= 1) return plan;
        SplitPlan cand = with_splits([&](int qb) { return (T[qb] + lo - 1) / lo; });
        return cand.chunk ? cand : plan;
    }
    if (!multiwave || base <= sms || base > 4LL * sms) return plan;
    // cost of an item beyond its key tiles and of the merge, in key steps
    // (measured: the D = 64 key step is about half as long as the D = 128 one)
    const double per_item = kernel_dim(D) == 64 ? FA_PLAN_ITEM_D64 : FA_PLAN_ITEM_D128;
    const double merge = kernel_dim(D) == 64 ? FA_PLAN_MERGE_D64 : FA_PLAN_MERGE_D128;
    if (!order_items(plan, S, causal)) return no_split(S);
    const double t0 = simulate_plan(plan, S, causal, bh, sms, per_item, merge);
    SplitPlan best = plan;
    double t_best = t0;
    // candidates that cannot beat the best so far (their work spread evenly
    // over the CTAs already takes longer) are not simulated
    auto consider = [&](const SplitPlan& cand) {
        if (!cand.chunk || cand.max_splits <= 1) return;
        double work = 0.0;
        for (int qb = 0; qb < nqb; ++qb) work += T[qb] + per_item * cand.ns[qb];
        const long long items = bh * cand.ctas_per_head;
        if (work * bh / static_cast<double>(std::min<long long>(items, sms)) + merge >= t_best) return;
        const double t = simulate_plan(cand, S, causal, bh, sms, per_item, merge);
        if (t < t_best) {
            t_best = t;
            best = cand;
        }
    };
    int tmax = 0;
    for (int qb = 0; qb < nqb; ++qb) tmax = std::max(tmax, T[qb]);
    int prev_ns0 = -1, prev_nsl = -1;   // (caps that split like the previous one are skipped)
    for (int cap = 1; cap < tmax; ++cap) {
        const int ns0 = (T[0] + cap - 1) / cap, nsl = (T[nqb - 1] + cap - 1) / cap;
        if (ns0 == prev_ns0 && nsl == prev_nsl && T[0] == T[nqb - 1]) continue;
        prev_ns0 = ns0;
        prev_nsl = nsl;
        consider(with_splits([&](int qb) { return (T[qb] + cap - 1) / cap; }));
    }
    int by_len[fa::kMaxSplitBlocks];   // blocks lightest first
    for (int qb = 0; qb < nqb; ++qb) by_len[qb] = qb;
    std::stable_sort(by_len, by_len + nqb, [&](int a, int b) { return T[a] < T[b]; });
    const int m_step = std::max(1, (nqb - 1) / 16);   // at most ~16 block counts
    for (int m = 1; m < nqb; m += m_step) {
        for (int n = 2; n <= 4; ++n) {
            bool light[fa::kMaxSplitBlocks] = {};
            for (int i = 0; i < m; ++i) light[by_len[i]] = true;
            consider(with_splits([&](int qb) { return light[qb] ? n : 1; }));
            consider(with_splits([&](int qb) { return light[qb] ? 1 : n; }));
        }
    }
    if (t_best > 0.92 * t0) return no_split(S);
    return best;
}

// Plans are cached per shape (host threads may call concurrently).
SplitPlan plan_split(int B, int H, int S, int D, bool causal, int sms, bool multiwave = true) {
    struct Entry { int B, H, S, kd, causal, sms; bool multiwave; SplitPlan plan; };
    static std::mutex mu;
    static Entry cache[32];
    static int used = 0, next = 0;
    const int kd = kernel_dim(D);
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry& e = cache[i];
            if (e.B == B && e.H == H && e.S == S && e.kd == kd && e.causal == int(causal) && e.sms == sms &&
                e.multiwave == multiwave)
                return e.plan;
        }
    }
    const SplitPlan plan = plan_split_uncached(B, H, S, D, causal, sms, multiwave);
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = Entry{B, H, S, kd, int(causal), sms, multiwave, plan};
    next = (next + 1) % 32;
    used = std::max(used, next == 0 ? 32 : next);
    return plan;
}

size_t workspace_bytes_for(const SplitPlan& plan, int B, int H, int S, int D_head) {
    if (plan.chunk == 0) return 0;
    const int D = kernel_dim(D_head);   // the partials have the kernel's width
    const size_t ntq = (S + fa::kBM - 1) / fa::kBM;
    const size_t slots = static_cast<size_t>(B) * H * ntq * plan.max_splits;
    return slots * (static_cast<size_t>(fa::kBM) * D + 2 * fa::kBM) * sizeof(float);
}

// What a call adds to the plain batched forward (one at a time).
struct Options {
    const int* cu_seqlens = nullptr;   // packed variable-length batch
    int total = 0;
    int win_left = -1, win_right = -1; // local attention
    bool dropout = false;              // attention dropout
    unsigned long long seed = 0;
    uint32_t drop_threshold = 0;
    float drop_inv_keep = 1.f;
    int drop_first_q = 0;              // test support: the first Q load is withheld
};

// Merge the partials of a split call (fa_combine_kernel), launched as a
// programmatic dependent of the main kernel: the launch gap is hidden.
template <int D, bool BF16>
int launch_combine(const fa::FwdParams& p, void* O, int B, int H, size_t ntq, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    constexpr int kThreads = fa::combine_threads(D);
    constexpr int kPerTile = fa::kBM / (kThreads / (D / 8));
    cfg.gridDim = dim3(static_cast<unsigned>(ntq * kPerTile),
                       static_cast<unsigned>(B) * static_cast<unsigned>(H));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fa::fa_combine_kernel<D, BF16>, p, O) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

template <int D, bool BF16, int NS, int RS, int FEAT>
int launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Hkv,
           int S, int Dh, int causal, float scale, cudaStream_t stream, const SplitPlan& plan,
           void* workspace, const Options& opt) {
    const int* cu_seqlens = opt.cu_seqlens;
    const int total = opt.total;
    auto kern = fa::fa_fwd_kernel<D, BF16, NS, RS, FEAT>;
    constexpr int kSmem = fa::SmemLayout<D, NS, RS>::kAlloc;
    // The dynamic shared-memory opt-in is per device; remember it per device.
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
    std::call_once(once[dev], [&] {
        attr_err[dev] =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    });
    if (attr_err[dev] != cudaSuccess) return FA_ERR_CUDA;

    // packed variable-length tensors are one batch of `total` rows
    const int mb = cu_seqlens ? 1 : B;
    const int ms = cu_seqlens ? total : S;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, Q, BF16, mb, ms, H, Dh, fa::kBM) || !make_map(&mk, K, BF16, mb, ms, Hkv, Dh, fa::kBN) ||
        !make_map(&mv, V, BF16, mb, ms, Hkv, Dh, fa::kBN) || !make_map(&mo, O, BF16, mb, ms, H, Dh, fa::kBM))
        return FA_ERR_CUDA;

    fa::FwdParams p;
    p.B = B;
    p.H = H;
    p.S = S;
    p.d_head = Dh;
    p.causal = causal ? 1 : 0;
    p.kv_group = H / Hkv;
    p.cu_seqlens = cu_seqlens;
    p.win_left = opt.win_left;
    p.win_right = opt.win_right;
    p.drop_first_q = opt.drop_first_q;
    p.drop_seed_lo = static_cast<uint32_t>(opt.seed & 0xffffffffull);
    p.drop_seed_hi = static_cast<uint32_t>(opt.seed >> 32);
    p.drop_threshold = opt.drop_threshold;
    p.drop_inv_keep = opt.drop_inv_keep;
    p.total = total;
    p.o_ptr = O;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.lse = LSE;
    const int rows_per_cta = fa::kQTiles * fa::kBM;
    p.nqb = (S + rows_per_cta - 1) / rows_per_cta;
    p.kv_chunk = plan.chunk;
    p.max_splits = plan.max_splits;
    const size_t ntq = (S + fa::kBM - 1) / fa::kBM;
    const size_t o_floats = static_cast<size_t>(B) * H * ntq * plan.max_splits * fa::kBM * D;
    p.ws_o = plan.chunk ? static_cast<float*>(workspace) : nullptr;
    p.ws_ml = plan.chunk ? static_cast<float*>(workspace) + o_floats : nullptr;
    if (plan.chunk) {
        std::copy(plan.item, plan.item + plan.ctas_per_head, p.split_item);
        std::copy(plan.ns, plan.ns + fa::kMaxSplitBlocks, p.block_splits);
    }
    // one CTA per SM, each running its share of the work items (at most one
    // CTA per item)
    const long long items = static_cast<long long>(B) * H * plan.ctas_per_head;
    p.items = static_cast<int>(items);
    const int sms = num_sms();
    const long long ctas = (sms > 0 && items > sms) ? sms : items;
    // Programmatic dependent launch: the CTAs may start (barrier and TMEM
    // set-up) while the previous kernel in the stream drains; the kernel
    // waits for it before its first load.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t mcfg = {};
    mcfg.gridDim = dim3(static_cast<unsigned>(ctas));
    mcfg.blockDim = dim3(fa::Roles<RS>::kThreads);
    mcfg.dynamicSmemBytes = kSmem;
    mcfg.stream = stream;
    mcfg.attrs = pdl;
    mcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&mcfg, kern, mq, mk, mv, mo, p) != cudaSuccess) return FA_ERR_CUDA;
    if (plan.chunk == 0) return FA_OK;

    return launch_combine<D, BF16>(p, O, B, H, ntq, stream);
}

int validate(const void* Q, const void* K, const void* V, void* O, const float* LSE, int B, int H,
             int S, int D, float scale, int dtype) {
    if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || S < 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (!supported_dim(D)) return FA_ERR_UNSUPPORTED;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                          reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O);
    if (mis & 15u) return FA_ERR_UNSUPPORTED;
    if (LSE != nullptr && (reinterpret_cast<uintptr_t>(LSE) & 3u)) return FA_ERR_UNSUPPORTED;
    // work items (query blocks of 256 rows times B*H) are numbered with an
    // int; a head holds at most 65535 query blocks
    const long long rows_per_cta = static_cast<long long>(fa::kQTiles) * fa::kBM;
    const long long nqb = (static_cast<long long>(S) + rows_per_cta - 1) / rows_per_cta;
    if (nqb > 65535) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * H * nqb > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// D in (128, 256]: one CTA per (head, 128-row query tile) at width 192 or
// 256, programmatic dependent launch as the main kernel.
template <int D, bool BF16, bool DROP>
int launch_wide(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                int Hkv, int S, int Dh, int causal, float scale, cudaStream_t stream, const SplitPlan& plan,
                void* workspace, const Options& opt) {
    auto kern = fa::fa_fwd_wide_kernel<D, BF16, DROP>;
    constexpr int kSmem = fa::WideSmem<D>::kAlloc;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    });
    if (attr_err[dev] != cudaSuccess) return FA_ERR_CUDA;
    // packed variable-length tensors are one batch of `total` rows
    const int mb = opt.cu_seqlens ? 1 : B;
    const int ms = opt.cu_seqlens ? opt.total : S;
    CUtensorMap mq, mk, mv, mo;
    // V is copied in pieces of kVRows keys
    if (!make_map(&mq, Q, BF16, mb, ms, H, Dh, fa::kBM) || !make_map(&mk, K, BF16, mb, ms, Hkv, Dh, fa::kBN) ||
        !make_map(&mv, V, BF16, mb, ms, Hkv, Dh, fa::WideSmem<D>::kVRows) ||
        !make_map(&mo, O, BF16, mb, ms, H, Dh, fa::kBM))
        return FA_ERR_CUDA;
    fa::FwdParams p = {};
    p.B = B;
    p.H = H;
    p.S = S;
    p.d_head = Dh;
    p.causal = causal ? 1 : 0;
    p.kv_group = H / Hkv;
    p.o_ptr = O;
    p.lse = LSE;
    p.cu_seqlens = opt.cu_seqlens;
    p.total = opt.total;
    p.win_left = opt.win_left;
    p.win_right = opt.win_right;
    p.drop_first_q = opt.drop_first_q;
    p.drop_seed_lo = static_cast<uint32_t>(opt.seed & 0xffffffffull);
    p.drop_seed_hi = static_cast<uint32_t>(opt.seed >> 32);
    p.drop_threshold = opt.drop_threshold;
    p.drop_inv_keep = opt.drop_inv_keep;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    const size_t ntq = (S + fa::kBM - 1) / fa::kBM;
    // split over keys: max_splits CTAs per query tile, partials in the
    // workspace, merged by fa_combine_kernel
    p.kv_chunk = plan.chunk;
    p.max_splits = plan.chunk ? plan.max_splits : 1;
    p.nqb = (S + fa::kQTiles * fa::kBM - 1) / (fa::kQTiles * fa::kBM);
    if (plan.chunk) {
        const size_t o_floats = static_cast<size_t>(B) * H * ntq * plan.max_splits * fa::kBM * D;
        p.ws_o = static_cast<float*>(workspace);
        p.ws_ml = static_cast<float*>(workspace) + o_floats;
        std::copy(plan.ns, plan.ns + fa::kMaxSplitBlocks, p.block_splits);
    }
    const long long ctas = static_cast<long long>(B) * H * ntq * p.max_splits;
    if (ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(fa::kWideThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, p) != cudaSuccess) return FA_ERR_CUDA;
    if (plan.chunk == 0) return FA_OK;
    return launch_combine<D, BF16>(p, O, B, H, ntq, stream);
}

int dispatch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Hkv,
             int S, int D, int causal, float scale, int dtype, cudaStream_t st, const SplitPlan& plan,
             void* ws, const Options& opt = Options()) {
    // <head dim, bf16, K/V ring slots, softmax threads per query row, feature>:
    // packed variable-length batches, local windows and dropout have kernel
    // variants of their own; the plain one compiles none of them
    const int feat = opt.cu_seqlens != nullptr ? fa::kPacked
                     : (opt.win_left >= 0 || opt.win_right >= 0) ? fa::kLocal
                     : opt.dropout ? fa::kDropout : fa::kPlain;
#define FA_ONE(D_, BF16_, NS_, RS_, F_) \
    launch<D_, BF16_, NS_, RS_, F_>(Q, K, V, O, LSE, B, H, Hkv, S, D, causal, scale, st, plan, ws, opt)
#define FA_LAUNCH(D_, BF16_, NS_, RS_)                                    \
    (feat == fa::kPacked    ? FA_ONE(D_, BF16_, NS_, RS_, fa::kPacked)    \
     : feat == fa::kLocal   ? FA_ONE(D_, BF16_, NS_, RS_, fa::kLocal)     \
     : feat == fa::kDropout ? FA_ONE(D_, BF16_, NS_, RS_, fa::kDropout)   \
                            : FA_ONE(D_, BF16_, NS_, RS_, fa::kPlain))
    const int kd = kernel_dim(D);
    if (kd > 128) {
        // every variant; only plain calls are split over keys
        if (feat != fa::kPlain && plan.chunk != 0) return FA_ERR_UNSUPPORTED;
        const bool drop = feat == fa::kDropout;
#define FA_WIDE(D_, BF16_)                                                                              \
    (drop ? launch_wide<D_, BF16_, true>(Q, K, V, O, LSE, B, H, Hkv, S, D, causal, scale, st, plan, ws, opt) \
          : launch_wide<D_, BF16_, false>(Q, K, V, O, LSE, B, H, Hkv, S, D, causal, scale, st, plan, ws, opt))
        if (dtype == FA_F16) return kd == 192 ? FA_WIDE(192, false) : FA_WIDE(256, false);
        return kd == 192 ? FA_WIDE(192, true) : FA_WIDE(256, true);
#undef FA_WIDE
    }
    if (dtype == FA_F16) {
        if (kd == 64) return FA_LAUNCH(64, false, kRingD64, kRowSplitD64);
        return FA_LAUNCH(128, false, kRingD128, kRowSplitD128);
    }
    if (kd == 64) return FA_LAUNCH(64, true, kRingD64, kRowSplitD64);
    return FA_LAUNCH(128, true, kRingD128, kRowSplitD128);
#undef FA_LAUNCH
#undef FA_ONE
}

}  // namespace

extern "C" {

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int S,
           int D, int causal, float scale, int dtype, fa_stream_t stream) {
    const int v = validate(Q, K, V, O, LSE, B, H, S, D, scale, dtype);
    if (v != FA_OK) return v;
    return dispatch(Q, K, V, O, LSE, B, H, H, S, D, causal, scale, dtype,
                    reinterpret_cast<cudaStream_t>(stream), SplitPlan{0, 1, (S + 255) / 256}, nullptr);
}

int fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
               int H_kv, int S, int D, int causal, float scale, int dtype, fa_stream_t stream) {
    const int v = validate(Q, K, V, O, LSE, B, H, S, D, scale, dtype);
    if (v != FA_OK) return v;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    return dispatch(Q, K, V, O, LSE, B, H, H_kv, S, D, causal, scale, dtype,
                    reinterpret_cast<cudaStream_t>(stream), SplitPlan{0, 1, (S + 255) / 256}, nullptr);
}

int fa_fwd_local(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int H_kv, int S, int D, int causal, int window_left, int window_right, float scale,
                 int dtype, fa_stream_t stream) {
    const int v = validate(Q, K, V, O, LSE, B, H, S, D, scale, dtype);
    if (v != FA_OK) return v;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
    Options opt;
    opt.win_left = window_left;
    opt.win_right = window_right;
    return dispatch(Q, K, V, O, LSE, B, H, H_kv, S, D, causal, scale, dtype,
                    reinterpret_cast<cudaStream_t>(stream), SplitPlan{0, 1, (S + 255) / 256}, nullptr, opt);
}

int fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                   int H_kv, int S, int D, int causal, double p_drop, unsigned long long seed,
                   float scale, int dtype, fa_stream_t stream) {
    const int v = validate(Q, K, V, O, LSE, B, H, S, D, scale, dtype);
    if (v != FA_OK) return v;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (!(p_drop >= 0.0 && p_drop < 1.0)) return FA_ERR_INVALID_ARG;
    Options opt;
    opt.dropout = true;
    opt.seed = seed;
    // keep iff the 16-bit draw >= floor(p * 2^16); the kernel compares it
    // in the upper half of a 32-bit word
    const double t = std::min(std::floor(p_drop * 65536.0), 65535.0);
    opt.drop_threshold = static_cast<uint32_t>(t) << 16;
    opt.drop_inv_keep = static_cast<float>(1.0 / (1.0 - p_drop));
    return dispatch(Q, K, V, O, LSE, B, H, H_kv, S, D, causal, scale, dtype,
                    reinterpret_cast<cudaStream_t>(stream), SplitPlan{0, 1, (S + 255) / 256}, nullptr, opt);
}

int fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                  const int* cu_seqlens, int B, int max_seqlen, int total, int H, int H_kv, int D,
                  int causal, float scale, int dtype, fa_stream_t stream) {
    // the shape checks of the batched call, on one batch of `total` rows
    const int v = validate(Q, K, V, O, LSE, 1, H, total, D, scale, dtype);
    if (v != FA_OK) return v;
    if (cu_seqlens == nullptr || B < 1 || max_seqlen < 1 || max_seqlen > total) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) return FA_ERR_UNSUPPORTED;
    const long long nqb = (static_cast<long long>(max_seqlen) + 255) / 256;
    if (static_cast<long long>(B) * H * nqb > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    Options opt;
    opt.cu_seqlens = cu_seqlens;
    opt.total = total;
    return dispatch(Q, K, V, O, LSE, B, H, H_kv, max_seqlen, D, causal, scale, dtype,
                    reinterpret_cast<cudaStream_t>(stream), SplitPlan{0, 1, static_cast<int>(nqb)},
                    nullptr, opt);
}

int fa_splitkv_workspace_size(int B, int H, int S, int D, int causal, size_t* bytes) {
    if (bytes == nullptr || B < 1 || H < 1 || S < 1) return FA_ERR_INVALID_ARG;
    if (!supported_dim(D)) return FA_ERR_UNSUPPORTED;
    const int sms = num_sms();
    if (sms <= 0) return FA_ERR_CUDA;
    *bytes = workspace_bytes_for(plan_split(B, H, S, D, causal != 0, sms), B, H, S, D);
    return FA_OK;
}

int fa_splitkv_launches(int B, int H, int S, int D, int causal) {
    if (B < 1 || H < 1 || S < 1 || !supported_dim(D)) return 0;
    return plan_split(B, H, S, D, causal != 0, num_sms()).chunk ? 2 : 1;
}

int fa_split_plan(int B, int H, int S, int D, int causal, int sms, int* splits, int max_blocks,
                  int* items_per_head) {
    if (B < 1 || H < 1 || S < 1 || D < 1 || sms < 1 || (splits == nullptr && max_blocks > 0))
        return FA_ERR_INVALID_ARG;
    const SplitPlan plan = plan_split(B, H, S, D, causal != 0, sms);
    const int nqb = (S + fa::kQTiles * fa::kBM - 1) / (fa::kQTiles * fa::kBM);
    for (int qb = 0; qb < std::min(nqb, max_blocks); ++qb)
        splits[qb] = plan.chunk && qb < fa::kMaxSplitBlocks ? plan.ns[qb] : 1;
    if (items_per_head != nullptr) *items_per_head = plan.ctas_per_head;
    return plan.chunk ? plan.max_splits : 1;
}

int fa_fwd_gqa_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                       int H, int H_kv, int S, int D, int causal, float scale, int dtype,
                       void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    const int v = validate(Q, K, V, O, LSE, B, H, S, D, scale, dtype);
    if (v != FA_OK) return v;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    const int sms = num_sms();
    if (sms <= 0) return FA_ERR_CUDA;
    const SplitPlan plan = plan_split(B, H, S, D, causal != 0, sms);
    const size_t need = workspace_bytes_for(plan, B, H, S, D);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return FA_ERR_INVALID_ARG;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 15u)) return FA_ERR_UNSUPPORTED;
    return dispatch(Q, K, V, O, LSE, B, H, H_kv, S, D, causal, scale, dtype,
                    reinterpret_cast<cudaStream_t>(stream), plan, workspace);
}

int fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                   int S, int D, int causal, float scale, int dtype, void* workspace,
                   size_t workspace_bytes, fa_stream_t stream) {
    return fa_fwd_gqa_splitkv(Q, K, V, O, LSE, B, H, H, S, D, causal, scale, dtype, workspace,
                              workspace_bytes, stream);
}

int fa_fwd_f16(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
               int S, int D, int causal, float scale, fa_stream_t stream) {
    return fa_fwd(Q, K, V, O, LSE, B, H, S, D, causal, scale, FA_F16, stream);
}

int fa_fwd_bf16(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                int S, int D, int causal, float scale, fa_stream_t stream) {
    return fa_fwd(Q, K, V, O, LSE, B, H, S, D, causal, scale, FA_BF16, stream);
}

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported shape, head dimension or alignment";
        case FA_ERR_CUDA: return "CUDA runtime or driver error";
        case FA_ERR_TIMEOUT: return "a device-side wait timed out";
        case FA_ERR_BAD_SEQLENS: return "a sequence offset was out of range (that sequence was skipped)";
        case FA_ERR_DEVICE_CHECK: return "a device-side invariant check failed (debug build)";
        default: return "unknown status";
    }
}

int fa_device_status(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, fa::g_fa_device_status, sizeof(int)) != cudaSuccess)
        return FA_ERR_CUDA;
    if (clear) {
        const int z = 0;
        if (cudaMemcpyToSymbol(fa::g_fa_device_status, &z, sizeof(int)) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return v;
}

int fa_last_device_status(fa_stream_t stream) {
    // pageable destination: the copy returns once it has landed, in stream order
    int v = 0;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyFromSymbolAsync(&v, fa::g_fa_device_status, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                  st) != cudaSuccess)
        return FA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
    return v;
}

int fa_selftest_timeout(const void* Q, const void* K, const void* V, void* O, int S, int D, int dtype,
                        fa_stream_t stream) {
    const int v = validate(Q, K, V, O, nullptr, 1, 1, S, D, 1.f, dtype);
    if (v != FA_OK) return v;
    Options opt;
    opt.drop_first_q = 1;
    return dispatch(Q, K, V, O, nullptr, 1, 1, 1, S, D, 0, D == 64 ? 0.125f : 0.08838835f, dtype,
                    reinterpret_cast<cudaStream_t>(stream), SplitPlan{0, 1, (S + 255) / 256}, nullptr, opt);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of fa_fwd_splitkv.
//
// Some callers cannot call cudaMalloc: a latency-critical loop that must not
// pay for cudaMalloc's implicit device synchronisation, a program whose device
// memory belongs to an allocator it cannot reach from this call site, or
// plain C code that links only this library.  For them the split-over-keys
// scratch lives in one file-scope device array, so a call needs no workspace
// argument and allocates nothing.  The array (kStaticWorkspaceBytes) is
// reserved on every GPU that loads this library until the process exits.
namespace {
constexpr size_t kStaticWorkspaceBytes = static_cast<size_t>(24) << 20;   // 24 MiB
}  // namespace

static __device__ __align__(256) unsigned char g_fa_static_workspace[kStaticWorkspaceBytes];

namespace {

// In host code `g_fa_static_workspace` only names a host-side stand-in for
// the symbol; its device address is looked up once per device, with that
// device current, on the first call made on it.
void* static_workspace_address(int* status) {
    static std::once_flag once[64];
    static void* address[64];
    static cudaError_t lookup[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *status = FA_ERR_CUDA;
        return nullptr;
    }
    std::call_once(once[dev], [&] {
        void* p = nullptr;
        lookup[dev] = cudaGetSymbolAddress(&p, g_fa_static_workspace);
        address[dev] = p;
    });
    if (lookup[dev] != cudaSuccess || address[dev] == nullptr) {
        *status = FA_ERR_CUDA;
        return nullptr;
    }
    return address[dev];
}

}  // namespace

extern "C" int fa_fwd_splitkv_static(const void* Q, const void* K, const void* V, void* O,
                                     float* LSE, int B, int H, int S, int D, int causal,
                                     float scale, int dtype, fa_stream_t stream) {
    const int v = validate(Q, K, V, O, LSE, B, H, S, D, scale, dtype);
    if (v != FA_OK) return v;
    const int sms = num_sms();
    if (sms <= 0) return FA_ERR_CUDA;
    // the one-wave plans only: the multi-wave ones need more scratch than the
    // array holds for the shapes they serve
    const SplitPlan plan = plan_split(B, H, S, D, causal != 0, sms, false);
    const size_t need = workspace_bytes_for(plan, B, H, S, D);
    if (need > kStaticWorkspaceBytes) return FA_ERR_UNSUPPORTED;
    // looked up on every call (free after the first), so that the first call
    // on a device does the lookup whether or not its shape is split
    int status = FA_OK;
    void* ws = static_workspace_address(&status);
    if (ws == nullptr) return status;
    return dispatch(Q, K, V, O, LSE, B, H, H, S, D, causal, scale, dtype,
                    reinterpret_cast<cudaStream_t>(stream), plan, ws);
}

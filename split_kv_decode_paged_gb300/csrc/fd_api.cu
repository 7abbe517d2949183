// fd_api.cu -- the C ABI of libfd (declared in include/fd_api.h): problem
// validation, the split-count cost model, TMA descriptor encoding and the
// kernel launches.  No device memory is allocated here.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <numeric>
#include <queue>
#include <vector>

#include "fd_internal.h"

namespace fd {

cudaError_t launch_decode_f16(const fd_problem &, const KernelShape &, const DecodeParams &, const CUtensorMap &,
                              const CUtensorMap &, int, size_t, cudaStream_t);
cudaError_t launch_decode_bf16(const fd_problem &, const KernelShape &, const DecodeParams &, const CUtensorMap &,
                               const CUtensorMap &, int, size_t, cudaStream_t);
cudaError_t launch_decode_e4m3(const fd_problem &, const KernelShape &, const DecodeParams &, const CUtensorMap &,
                               const CUtensorMap &, int, size_t, cudaStream_t);
cudaError_t decode_occupancy_f16(const fd_problem &, const KernelShape &, size_t, int *);
cudaError_t decode_occupancy_bf16(const fd_problem &, const KernelShape &, size_t, int *);
cudaError_t decode_occupancy_e4m3(const fd_problem &, const KernelShape &, size_t, int *);
size_t decode_smem_f16(const fd_problem &, const KernelShape &, int, bool);
size_t decode_smem_bf16(const fd_problem &, const KernelShape &, int, bool);
size_t decode_smem_e4m3(const fd_problem &, const KernelShape &, int, bool);

KernelShape kernel_shape(const fd_problem &p, int tile_tokens, int fold, int ctas_per_sm) {
    KernelShape ks;
    // 256-token stages: E4M3 only, with pages of >= 32 tokens (at most
    // kMaxBoxesPerTile boxes per stage).
    const bool t256 = tile_tokens == 256 && p.kv_dtype == FD_E4M3 &&
                      std::gcd(p.page_size, 256) * kMaxBoxesPerTile >= 256;
    const int tile = tile_tokens == 64 ? 64 : (t256 ? 256 : 128);
    if (tile == 64) {
        ks.consumer_warps = 4;
        ks.subtiles = 1;
    } else if (tile == 128 && ctas_per_sm >= 2 && p.kv_dtype == FD_E4M3) {
        // 4 consumer warps, 32 tokens each per 128 (two sub-tiles sharing one
        // online-softmax step): the register budget of two CTAs per SM.
        ks.consumer_warps = 4;
        ks.subtiles = 2;
    } else {
        // 8 consumer warps, 16 tokens each per 128 (one sub-tile; E4M3 with
        // 256-token stages: two).
        ks.consumer_warps = 8;
        ks.subtiles = tile / 128;
    }
    ks.tile = ks.consumer_warps * ks.subtiles * kTokensPerWarp;
    ks.nt = (p.Hq / p.Hkv) * fold <= 8 ? 1 : 2;
    return ks;
}

size_t decode_smem_bytes(const fd_problem &p, const KernelShape &ks, int stages, bool scr_in_stage) {
    switch (p.kv_dtype) {
    case FD_F16: return decode_smem_f16(p, ks, stages, scr_in_stage);
    case FD_BF16: return decode_smem_bf16(p, ks, stages, scr_in_stage);
    default: return decode_smem_e4m3(p, ks, stages, scr_in_stage);
    }
}

cudaError_t decode_occupancy(const fd_problem &p, const KernelShape &ks, size_t smem, int *blocks) {
    switch (p.kv_dtype) {
    case FD_F16: return decode_occupancy_f16(p, ks, smem, blocks);
    case FD_BF16: return decode_occupancy_bf16(p, ks, smem, blocks);
    default: return decode_occupancy_e4m3(p, ks, smem, blocks);
    }
}

cudaError_t launch_decode(const fd_problem &p, const KernelShape &ks, const DecodeParams &dp, const CUtensorMap &tmk,
                          const CUtensorMap &tmv, int grid, size_t smem, cudaStream_t stream) {
    switch (p.kv_dtype) {
    case FD_F16: return launch_decode_f16(p, ks, dp, tmk, tmv, grid, smem, stream);
    case FD_BF16: return launch_decode_bf16(p, ks, dp, tmk, tmv, grid, smem, stream);
    default: return launch_decode_e4m3(p, ks, dp, tmk, tmv, grid, smem, stream);
    }
}

}  // namespace fd

using namespace fd;

namespace {

constexpr int kMaxStages = 8;
constexpr int kMaxQLen = 64;  // query tokens per sequence (multi-token mode)
constexpr int kMinStages = 2;
constexpr int kSmallGridItemTokens = 1024;  // small grids: two CTAs per SM for items up to this long
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s limit on any device-side wait
// Cost-model constants (in token-times of one CTA): fixed cost of one work
// item (epilogue + pipeline hand-over) and the relative margin within which
// fewer splits are preferred.
constexpr double kItemOverheadTokens = 48.0;
// Extra CTA time of an item of a split sequence: publishing its partial
// state and the fused merge, measured at ~1.6 us, i.e. the bytes one CTA
// streams in that time (~45 GB/s per CTA).
constexpr double kSplitPublishBytes = 73728.0;
constexpr int kDefaultSplitMarginPct = 2;
// Below this many attended tokens per work item on average (and with enough
// items), the planner runs two CTAs per SM; for 16-bit K/V the higher figure
// applies when the default shape has lost pipeline depth to large dispatch
// tables (measured crossovers on GB300: ~700 and above 1024 tokens).  With
// TMA boxes of at most 4 KB (16-token pages at D = 128, up to 32-token pages
// at D = 64) one producer per SM issues them too slowly, and two CTAs (three
// stages each, their epilogue scratch in a stage) win up to 4096 tokens per
// item (same GPU, 256-1024 sequences, 8 KV heads: 16-token pages, D = 128,
// -3.5% at 1024 tokens, -0.7% at 4096; D = 64, 2048 tokens, -24%; 64-token
// pages, D = 128: +1%, so left to the other figures).  E4M3 K/V switch
// below 2048 tokens per item when the default shape has 256-token stages,
// and always otherwise (16-token pages or very large batches, where one
// producer per SM issuing 2 KB boxes is the limit).
constexpr double kShortItemTokens = 1024.0;
constexpr double kShortItemTokensShallow = 1280.0;
constexpr double kShortItemTokensSmallBox = 4096.0;
constexpr double kShortItemTokensE4m3 = 2048.0;

// Wait limit (>= 0; 0 = kTimeoutNs) and the stall test hook: off, or a
// role of 1 or 2 with an idle time of at most one second.
bool hooks_valid(int timeout_us, int stall_us, int stall_role) {
    if (timeout_us < 0 || stall_us < 0 || stall_us > 1000000) return false;
    if (stall_role < 0 || stall_role > 2) return false;
    return stall_role == 0 ? stall_us == 0 : stall_us > 0;
}

int elem_bytes(fd_dtype t) { return t == FD_E4M3 ? 1 : (t == FD_F32 ? 4 : 2); }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

fd_status validate_problem(const fd_problem *p) {
    if (!p) return FD_ERR_INVALID_ARG;
    if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->D < 1 || p->page_size < 1 || p->max_blocks_per_seq < 1 ||
        p->num_pages < 1)
        return FD_ERR_INVALID_ARG;
    if (p->Hq % p->Hkv != 0) return FD_ERR_INVALID_ARG;
    if (p->page_size % 16 != 0) return FD_ERR_INVALID_ARG;
    if (p->q_dtype != FD_F16 && p->q_dtype != FD_BF16) return FD_ERR_UNSUPPORTED;
    if (p->kv_dtype == FD_E4M3) {
        // q may be f16 or bf16
    } else if (p->kv_dtype != p->q_dtype) {
        return FD_ERR_UNSUPPORTED;
    }
    if (p->out_dtype != p->q_dtype && p->out_dtype != FD_F32) return FD_ERR_UNSUPPORTED;
    if (p->D != 64 && p->D != 128) return FD_ERR_UNSUPPORTED;
    if (p->B > kMaxBatch) return FD_ERR_UNSUPPORTED;
    if ((long long)p->page_size * p->max_blocks_per_seq > (1LL << 30)) return FD_ERR_UNSUPPORTED;
    return FD_OK;
}

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;     // per CTA (opt-in maximum)
    int smem_per_sm = 0;    // per SM
    int smem_reserved = 0;  // set aside per resident CTA
};

fd_status device_info(DeviceInfo &di) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FD_ERR_CUDA;
    static std::mutex mu;
    static std::vector<DeviceInfo> cache;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1);
    if (cache[dev].sms == 0) {
        DeviceInfo d;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FD_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
            return FD_ERR_CUDA;
        cache[dev] = d;
    }
    di = cache[dev];
    return FD_OK;
}

int round_up(long long x, int a) { return (int)(((x + a - 1) / a) * a); }

// Greedy list-scheduling estimate of the busiest CTA (in token-times) when
// the items of chunk length C are handed out to P CTAs in the kernel's
// dispatch order: every full chunk first, then each sequence's partial
// chunk, longest first (Hkv items per chunk).  Every item costs item_ovh
// more, and every item of a split sequence (L > C) split_ovh more again.
double makespan(const std::vector<int> &lens, int Hkv, int C, int P, double item_ovh, double split_ovh) {
    std::vector<double> items;
    std::vector<std::pair<int, double>> tails;
    for (int L : lens) {
        const double extra = L > C ? split_ovh : 0.0;
        for (int s = 0; s < L / C; ++s) items.push_back(C + extra);
        if (L == 0 || L % C) tails.push_back({L % C, extra});
    }
    std::stable_sort(tails.begin(), tails.end(), [](const std::pair<int, double> &a, const std::pair<int, double> &b) {
        return a.first > b.first;
    });
    for (const auto &t : tails) items.push_back(t.first + t.second);
    std::priority_queue<double, std::vector<double>, std::greater<double>> q;
    for (int i = 0; i < P; ++i) q.push(0.0);
    double worst = 0.0;
    for (double len : items) {
        for (int h = 0; h < Hkv; ++h) {
            double t = q.top();
            q.pop();
            t += len + item_ovh;
            worst = std::max(worst, t);
            q.push(t);
        }
    }
    return worst;
}

// The pages' split rule (lpnh.cn "进阶突破": a cost model over batch, heads,
// length and SM count, no split for short sequences; "Inference Cookbook"
// §6.3: no split when the batch already fills the SMs, otherwise the fewest
// splits whose efficiency is close to the best).  Returns the chunk length.
int choose_chunk(const std::vector<int> &lens, const fd_problem &p, int P, int tile, double margin) {
    const int maxL = *std::max_element(lens.begin(), lens.end());
    const int G = p.Hq / p.Hkv;
    if (maxL <= 2 * kMinChunkTokens) return std::max(tile, round_up(std::max(maxL, 1), tile));
    const long long W = (long long)p.B * p.Hkv;
    std::vector<int> cand;
    for (int s = 1; s <= 64; ++s) cand.push_back(s);
    for (int k = 1; k <= 8; ++k) cand.push_back((int)((k * (long long)P + W - 1) / W));
    std::sort(cand.begin(), cand.end());
    cand.erase(std::unique(cand.begin(), cand.end()), cand.end());
    struct Opt { int S, C; double cost; };
    std::vector<Opt> opts;
    int lastC = -1;
    for (int S : cand) {
        if (S < 1 || S > kMaxSplits) continue;
        const int C = std::max(tile, round_up((maxL + S - 1) / S, tile));
        if (C == lastC) continue;
        if (S > 1 && C < kMinChunkTokens) break;
        lastC = C;
        long long items = 0;
        for (int L : lens) items += (long long)(L == 0 ? 1 : (L + C - 1) / C) * p.Hkv;
        if (S > 1 && items > 16LL * P) continue;
        const int nmax = (maxL + C - 1) / C;
        const double split_ovh = kSplitPublishBytes / (2.0 * p.D * elem_bytes(p.kv_dtype));
        double cost = makespan(lens, p.Hkv, C, P, kItemOverheadTokens, split_ovh);
        if (nmax > 1) cost += 0.5 * G * nmax;  // merge of nmax partials by one CTA
        opts.push_back({S, C, cost});
    }
    if (opts.empty()) return std::max(tile, round_up(maxL, tile));
    double best = opts[0].cost;
    for (auto &o : opts) best = std::min(best, o.cost);
    // Largest chunk (fewest splits) within the margin of the best.
    int bestC = opts[0].C;
    for (auto &o : opts)
        if (o.cost <= best * (1.0 + margin)) { bestC = o.C; break; }
    return bestC;
}

// ------------------------------------------------------- tensor map encoding
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// K or V pool viewed as 5-D (d within a swizzle span, slot, span index,
// kvh, page): one box = `boxr` token rows x all of D for one KV head, landing
// in shared memory as [span][row][span bytes] so each span is one swizzled
// region (a span is 128 bytes, or the whole row when the row is shorter).
bool encode_pool_map(CUtensorMap *map, const void *pool, const fd_problem &p, int boxr) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int e = elem_bytes(p.kv_dtype);
    const int rb = p.D * e;
    const int span = rb > 128 ? 128 : rb;
    const int nspan = rb / span;
    cuuint64_t dims[5] = {(cuuint64_t)(span / e), (cuuint64_t)p.page_size, (cuuint64_t)nspan, (cuuint64_t)p.Hkv,
                          (cuuint64_t)p.num_pages};
    cuuint64_t strides[4] = {(cuuint64_t)rb * p.Hkv, (cuuint64_t)span, (cuuint64_t)rb,
                             (cuuint64_t)rb * p.Hkv * p.page_size};
    cuuint32_t box[5] = {(cuuint32_t)(span / e), (cuuint32_t)boxr, (cuuint32_t)nspan, 1u, 1u};
    cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    const CUtensorMapDataType dt = e == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    const CUtensorMapSwizzle sw = span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    // L2 promotion no wider than one row: a wider promotion also fetches the
    // neighbouring KV head's row, which another CTA reads at another time.
    const CUtensorMapL2promotion l2p = rb >= 256   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                       : rb >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                   : CU_TENSOR_MAP_L2_PROMOTION_L2_64B;
    CUresult r = fn(map, dt, 5, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    l2p, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int fd_api_version(void) { return FD_API_VERSION; }

const char *fd_status_string(fd_status s) {
    switch (s) {
    case FD_OK: return "ok";
    case FD_ERR_INVALID_ARG: return "invalid argument";
    case FD_ERR_UNSUPPORTED: return "unsupported problem";
    case FD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FD_ERR_BAD_PAGE: return "block-table entry out of range";
    case FD_ERR_CUDA: return "CUDA error";
    case FD_ERR_CAPACITY: return "sequence length above the plan capacity";
    case FD_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

fd_status fd_status_from_device(int32_t w) {
    if (w & FD_DEV_TIMEOUT) return FD_ERR_TIMEOUT;
    if (w & FD_DEV_BAD_PAGE) return FD_ERR_BAD_PAGE;
    if (w & FD_DEV_CAPACITY) return FD_ERR_CAPACITY;
    return FD_OK;
}

fd_status fd_plan(const fd_problem *problem, const int32_t *seq_lens_host, const fd_plan_options *options,
                  fd_plan_t *plan) {
    if (!plan || !seq_lens_host) return FD_ERR_INVALID_ARG;
    fd_status st = validate_problem(problem);
    if (st != FD_OK) return st;
    fd_plan_options opt = {0, 0, 1, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    if (options) opt = *options;
    if (opt.num_splits < 0 || opt.num_sms < 0 || opt.max_seq_len < 0 || opt.ctas_per_sm < 0 || opt.ctas_per_sm > 8 ||
        opt.split_margin_pct < 0 || opt.split_margin_pct > 100 ||
        (opt.tile_tokens != 0 && opt.tile_tokens != 64 && opt.tile_tokens != 128 && opt.tile_tokens != 256) ||
        !hooks_valid(opt.timeout_us, opt.debug_stall_us, opt.debug_stall_role) || opt.q_len < 0 ||
        opt.q_len > kMaxQLen)
        return FD_ERR_INVALID_ARG;
    const int q_len = std::max(1, opt.q_len);
    if (q_len > 1 && opt.shared_kv) return FD_ERR_UNSUPPORTED;
    if ((long long)problem->B * q_len > kMaxBatch) return FD_ERR_UNSUPPORTED;
    // shared_kv: every q sequence attends KV row 0 (one block-table row, one
    // seq_lens entry): the B*G q rows of a KV head are sliced into items.
    // q_len > 1: the q_len query tokens of a sequence fold onto its KV row.
    const int fold = opt.shared_kv ? problem->B : q_len;
    const int kv_rows = opt.shared_kv ? 1 : problem->B;
    const double margin = (opt.split_margin_pct > 0 ? opt.split_margin_pct : kDefaultSplitMarginPct) / 100.0;
    const fd_problem &p = *problem;
    std::vector<int> lens(kv_rows);
    long long maxL = 0;
    for (int b = 0; b < kv_rows; ++b) {
        if (seq_lens_host[b] < 0) return FD_ERR_INVALID_ARG;
        lens[b] = seq_lens_host[b];
        maxL = std::max<long long>(maxL, lens[b]);
    }
    const long long capL = std::max<long long>(maxL, opt.max_seq_len);
    // shared memory of the dispatch tables follows the KV rows
    fd_problem pm = p;
    pm.B = kv_rows;
    if (capL > (long long)p.page_size * p.max_blocks_per_seq) return FD_ERR_INVALID_ARG;

    // The device is queried when present; planning for an explicit SM count
    // also works on a host without a GPU (shared memory then assumes GB300's
    // 227 KB per CTA, 228 KB per SM, 1 KB reserved per CTA).
    DeviceInfo di;
    int sms = opt.num_sms;
    st = device_info(di);
    const bool have_dev = st == FD_OK;
    if (!have_dev) {
        di.smem_optin = 232448;
        di.smem_per_sm = 233472;
        di.smem_reserved = 1024;
    }
    if (sms == 0) {
        if (!have_dev) return st;
        sms = di.sms;
    }
    // Dynamic shared memory one CTA may take when cps CTAs share an SM.
    auto smem_limit = [&](int cps) -> long long {
        if (cps <= 1) return di.smem_optin;
        return std::min<long long>(di.smem_optin, (di.smem_per_sm - (long long)cps * di.smem_reserved) / cps);
    };

    // One candidate kernel shape: stage size, CTAs per SM, chunk length,
    // partial slots, work items and the deepest pipeline that fits.
    struct Shape {
        KernelShape ks;
        int cps = 1, nhg = 1, C = 0, slots = 0, stages = 0;
        bool scr_in_stage = false;
        size_t smem = 0;
        long long items = 0;
    };
    auto make_shape = [&](int tile_opt, int cps, Shape &sh, int force_splits = 0) -> bool {
        sh.ks = kernel_shape(p, tile_opt, fold, cps);
        sh.cps = cps;
        const int tile = sh.ks.tile;
        const int qrows = 8 * sh.ks.nt;
        sh.nhg = ((p.Hq / p.Hkv) * fold + qrows - 1) / qrows;
        fd_problem pk = p;  // the KV side of the problem: kv_rows rows, nhg items per KV head
        pk.B = kv_rows;
        pk.Hkv = p.Hkv * sh.nhg;
        const int P = sms * cps;
        int C;
        const int S_opt = force_splits > 0 ? force_splits : opt.num_splits;
        if (S_opt > 0) {
            const int S = std::min(S_opt, kMaxSplits);
            C = std::max(tile, round_up((std::max<long long>(maxL, 1) + S - 1) / S, tile));
        } else {
            C = choose_chunk(lens, pk, P, tile, margin);
        }
        int slots = (int)std::max<long long>(1, (capL + C - 1) / C);
        if (slots > kMaxSplits) {
            C = std::max(tile, round_up((capL + kMaxSplits - 1) / kMaxSplits, tile));
            slots = (int)std::max<long long>(1, (capL + C - 1) / C);
        }
        sh.C = C;
        sh.slots = slots;
        sh.items = 0;
        for (int L : lens) sh.items += (long long)(L == 0 ? 1 : (L + C - 1) / C) * p.Hkv * sh.nhg;
        sh.stages = 0;
        sh.scr_in_stage = false;
        for (int s = kMaxStages; s >= kMinStages; --s) {
            const size_t need = decode_smem_bytes(pm, sh.ks, s, false);
            if ((long long)need <= smem_limit(cps)) {
                sh.stages = s;
                sh.smem = need;
                break;
            }
        }
        // The epilogue scratch in the item's last stage, where that makes
        // room for another stage.  Measured on GB300 (same GPU): four causal
        // query tokens, two 8-head tiles, 2 -> 3 stages -12%; GQA groups of
        // 16 -9.5%; one 4096-token sequence of 32 MHA heads on two CTAs per
        // SM -6.6%; 1024 sequences of 256-1024 tokens -3.7%.  With the stage
        // count unchanged it only costs (the tiny one-item call +0.7 us).
        // E4M3: only the two-CTA shape with 2 KB boxes (16-token pages):
        // 512-768 short sequences -6 to -9%; with 8-16 KB boxes the held
        // stage delays the next item's first copies (+3 to +8%), and 3
        // instead of 2 256-token stages with two head tiles measured 9% slower.
        const bool scr_ok = p.kv_dtype != FD_E4M3 || (long long)std::gcd(p.page_size, sh.ks.tile) * p.D <= 2048;
        for (int s = kMaxStages; scr_ok && s > std::max(sh.stages, kMinStages - 1); --s) {
            const size_t need = decode_smem_bytes(pm, sh.ks, s, true);
            if (need > 0 && (long long)need <= smem_limit(cps)) {
                sh.stages = s;
                sh.smem = need;
                sh.scr_in_stage = true;
                break;
            }
        }
        return sh.stages > 0;
    };

    // Default shape.  E4M3 pools take 256-token stages (8 consumer warps x 2
    // sub-tiles) when the pages allow them and three stages fit (two suffice
    // with two 8-head tiles: measured on GB300 with 32 to 128-token pages and
    // G = 12 or 16, two 256-token stages take 1-7% less time than five
    // 128-token ones); otherwise 128 (16-bit K/V: always 128).
    const int cps_opt = opt.ctas_per_sm > 0 ? opt.ctas_per_sm : 1;
    int tile_opt = opt.tile_tokens;
    if (q_len > 1) {
        // several causal query tokens per sequence: one CTA per SM, 128-token
        // stages of 8 consumer warps (the shape built with the causal limits)
        if ((opt.tile_tokens != 0 && opt.tile_tokens != 128) || cps_opt != 1) return FD_ERR_UNSUPPORTED;
        tile_opt = 128;
    }
    if (tile_opt == 0 && p.kv_dtype == FD_E4M3) {
        const KernelShape k256 = kernel_shape(p, 256, fold, cps_opt);
        const int need = k256.nt == 2 && cps_opt == 1 ? 2 : 3;
        if (k256.tile == 256 && (long long)decode_smem_bytes(pm, k256, need, false) <= smem_limit(cps_opt)) tile_opt = 256;
    }
    Shape sh;
    if (!make_shape(tile_opt, cps_opt, sh)) return FD_ERR_UNSUPPORTED;
    // Many short work items: two CTAs per SM with 64-token stages, so one
    // CTA streams while the other is between items (epilogue, next claim,
    // page ids).  Taken when the shape is left to the planner, the average
    // item attends fewer tokens than the threshold, there are enough items
    // for both CTAs of every SM, and two CTAs of that shape fit on an SM.
    if (q_len == 1 && opt.tile_tokens == 0 && opt.ctas_per_sm == 0 && sh.items >= 4LL * sms) {
        long long tok = 0;
        for (int L : lens) tok += L;
        const double mean_item = (double)tok * p.Hkv * sh.nhg / (double)sh.items;
        double limit;
        if (p.kv_dtype == FD_E4M3)
            limit = sh.ks.tile < 256 ? INFINITY : kShortItemTokensE4m3;
        else if ((long long)std::gcd(p.page_size, sh.ks.tile) * p.D * 2 <= 4096)
            limit = kShortItemTokensSmallBox + 1.0;  // up to and including 4096 tokens
        else
            limit = sh.stages < 3 ? kShortItemTokensShallow : kShortItemTokens;
        // E4M3: 128-token stages of 4 warps x 2 sub-tiles; 16-bit: 64-token stages.
        const int tile2 = p.kv_dtype == FD_E4M3 ? 128 : 64;
        Shape s2;
        if (mean_item < limit && make_shape(tile2, 2, s2)) {
            // Register budget of two 5-warp CTAs: three warps share one SM
            // sub-partition's 16K registers, so at most 168 per thread.  Without
            // a device, the shapes measured within it: one 8-head tile, or two
            // at D = 64 for 16-bit K/V.
            bool fits = s2.ks.nt == 1 || (p.D == 64 && p.kv_dtype != FD_E4M3);
            if (have_dev) {
                int blocks = 0;
                fits = decode_occupancy(p, s2.ks, s2.smem, &blocks) == cudaSuccess && blocks >= 2;
                cudaGetLastError();
            }
            if (fits) sh = s2;
        }
    }
    // Small grids: fewer work items than SMs leave SMs idle and each CTA's
    // start-up, ramp and tail exposed.  Two CTAs per SM with the most splits
    // whose items still fit the 2 x SMs slots halve the items and double the
    // streams; taken when the items stay short (at most kSmallGridItemTokens)
    // or the TMA boxes are small (at most 2 KB: one producer issues them too
    // slowly to keep an SM busy).  Measured on GB300 (same GPU, marginal time
    // per L2-flushed call): one sequence of 32 MHA heads, f16, 16-token pages,
    // D = 128: 2048 tokens -9.2%, 4096 tokens -2.2%, 16384 tokens +7% when
    // forced (so left alone by the item-length test); D = 64, 8192 tokens
    // (2 KB boxes) -16.6%; two sequences of 16 heads, 4096 tokens -0.6%.
    // Chunks keep the planner's floor (sequences of at most 2 x kMinChunkTokens
    // are not split, nor cut below kMinChunkTokens).
    // E4M3 K/V (128-token stages of 4 warps x 2 sub-tiles, same GPU): one
    // sequence of 32 MHA heads, 16-token pages, 2048 / 4096 tokens -9.6% /
    // -19%; 128-token pages, 4096 tokens -10%; two sequences of 16 heads,
    // 64-token pages, 8192 tokens -3%.
    // One sequence whose default plan leaves the busiest CTA two or more
    // items while at most 80% of the slots of its waves hold one (its equal
    // items cannot balance: e.g. 320 items on 152 SMs, 3 rounds for an average
    // of 2.1) is planned the same way, when its boxes are at most 2 KB or,
    // for 16-bit K/V, the two-CTA items keep at least 768 tokens.  Same GPU:
    // 32 MHA heads over 8192 f16 tokens, 16/32/64/128-token pages, 10 splits
    // on one CTA per SM 29.3-30.1 us, 9 splits (910 tokens) on two 26.5-26.8
    // us; E4M3 with 2 KB boxes (16 heads, 16-token pages at D = 128, 32-token
    // pages at D = 64) -6.3% / -2.4%; left alone: 16 f16 heads over 8192
    // tokens (19 splits of 431 on two CTAs, +1.8% to -6.4% by page size and
    // D) and E4M3 with 8-16 KB boxes (16 heads, 16384 tokens, +0.3 / +1.4%).
    bool medium = false;
    if (kv_rows == 1 && sh.items >= sms) {
        const long long waves = (sh.items + sms - 1) / sms;
        medium = waves >= 2 && (double)sh.items <= 0.8 * (double)(waves * sms);
    }
    if (q_len == 1 && opt.tile_tokens == 0 && opt.ctas_per_sm == 0 && opt.num_splits == 0 && sh.cps == 1 &&
        (sh.items < sms || medium) && maxL > 2 * kMinChunkTokens) {
        const int tile2 = p.kv_dtype == FD_E4M3 ? 128 : 64;
        int best_S = 0;
        for (int S = std::min(kMaxSplits, 2 * sms); S >= 1 && best_S == 0; --S) {
            Shape t;
            if (make_shape(tile2, 2, t, S) && t.items <= 2LL * sms && (t.slots == 1 || t.C >= kMinChunkTokens))
                best_S = S;
        }
        Shape s2;
        if (best_S > 0 && make_shape(tile2, 2, s2, best_S) && (s2.items > sh.items || (medium && s2.items >= sms))) {
            long long tok = 0;
            for (int L : lens) tok += L;
            const double mean_item = (double)tok * p.Hkv * s2.nhg / (double)s2.items;
            const int boxr2 = std::gcd(p.page_size, s2.ks.tile);
            const long long box_bytes = (long long)boxr2 * p.D * (p.kv_dtype == FD_E4M3 ? 1 : 2);
            bool fits = s2.ks.nt == 1 || (p.D == 64 && p.kv_dtype != FD_E4M3);
            if (have_dev) {
                int blocks = 0;
                fits = decode_occupancy(p, s2.ks, s2.smem, &blocks) == cudaSuccess && blocks >= 2;
                cudaGetLastError();
            }
            const bool medium_ok =
                !medium || box_bytes <= 2048 || (p.kv_dtype != FD_E4M3 && mean_item >= 768.0);
            if (fits && medium_ok && (mean_item <= kSmallGridItemTokens || box_bytes <= 2048)) sh = s2;
        }
    }
    const KernelShape ks = sh.ks;
    const int tile = ks.tile;
    const int nhg = sh.nhg;
    const int P = sms * sh.cps;
    const int C = sh.C;
    const int slots = sh.slots;
    const long long items = sh.items;
    const int stages = sh.stages;
    const size_t smem = sh.smem;

    std::memset(plan, 0, sizeof(*plan));
    plan->problem = p;
    plan->problem.B = kv_rows * fold;  // query rows
    plan->q_len = q_len;
    plan->num_splits = slots;
    plan->chunk_tokens = C;
    plan->tile_tokens = tile;
    plan->capacity_tokens = slots * C;
    plan->grid_ctas = (int)std::max<long long>(1, std::min<long long>(P, items));
    plan->num_sms = sms;
    plan->fuse_merge = opt.fuse_merge ? 1 : 0;
    plan->stages = stages;
    plan->scratch_in_stage = sh.scr_in_stage ? 1 : 0;
    plan->smem_bytes = (int)smem;
    plan->work_items_hint = items;
    plan->kv_rows = kv_rows;
    plan->row_fold = fold;
    plan->head_subgroups = nhg;
    plan->ctas_per_sm = sh.cps;
    plan->timeout_us = opt.timeout_us;
    plan->debug_stall_us = opt.debug_stall_us;
    plan->debug_stall_role = opt.debug_stall_role;
    const size_t rows = (size_t)plan->problem.B * p.Hq;
    size_t off = 0;
    plan->ws_partial_o = off;
    off += align256(slots > 1 ? rows * slots * p.D * sizeof(float) : 0);
    plan->ws_partial_md = off;
    off += align256(slots > 1 ? 2 * rows * slots * sizeof(float) : 0);
    plan->ws_counters = off;
    off += align256(((size_t)kv_rows * p.Hkv * nhg + 2) * sizeof(int));
    plan->workspace_bytes = off;
    return FD_OK;
}

}  // extern "C"

namespace {

fd_status decode_impl(const fd_plan_t *plan, const void *q, const void *k_pages, const void *v_pages,
                      const float *k_scale, const float *v_scale, const int32_t *block_table,
                      const int32_t *seq_lens, const fd_decode_extras *ex, void *out, float *lse, void *workspace,
                      size_t workspace_bytes, int32_t *status_dev, void *stream) {
    if (!plan) return FD_ERR_INVALID_ARG;
    const fd_problem &p = plan->problem;
    fd_status st = validate_problem(&p);
    if (st != FD_OK) return st;
    if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out || !workspace) return FD_ERR_INVALID_ARG;
    const bool fp8 = p.kv_dtype == FD_E4M3;
    if (fp8 != (k_scale != nullptr) || fp8 != (v_scale != nullptr)) return FD_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(workspace, 256) || (lse && !aligned(lse, 4)) || (k_scale && !aligned(k_scale, 4)) ||
        (v_scale && !aligned(v_scale, 4)) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return FD_ERR_INVALID_ARG;
    if (workspace_bytes < plan->workspace_bytes) return FD_ERR_WORKSPACE_TOO_SMALL;
    const int fold = plan->row_fold;
    if (fold < 1 || plan->kv_rows < 1 || plan->kv_rows * fold != p.B || plan->head_subgroups < 1) return FD_ERR_INVALID_ARG;
    const int q_len = std::max(1, plan->q_len);
    if (q_len > kMaxQLen || (q_len > 1 && fold != q_len)) return FD_ERR_INVALID_ARG;
    if (fold > 1 && ex && (ex->cache_batch_idx || ex->cache_leftpad)) return FD_ERR_UNSUPPORTED;
    if (plan->ctas_per_sm < 0 || plan->ctas_per_sm > 8) return FD_ERR_INVALID_ARG;
    const KernelShape ks = kernel_shape(p, plan->tile_tokens, fold, std::max(1, plan->ctas_per_sm));
    if (q_len > 1 && !(ks.consumer_warps == 8 && ks.subtiles == 1)) return FD_ERR_UNSUPPORTED;
    if (plan->head_subgroups != ((p.Hq / p.Hkv) * fold + 8 * ks.nt - 1) / (8 * ks.nt)) return FD_ERR_INVALID_ARG;
    if (plan->tile_tokens != ks.tile || plan->chunk_tokens < ks.tile || plan->chunk_tokens % ks.tile != 0 ||
        plan->num_splits < 1 || plan->num_splits > kMaxSplits || plan->stages < kMinStages ||
        plan->stages > kMaxStages || plan->grid_ctas < 1 ||
        !hooks_valid(plan->timeout_us, plan->debug_stall_us, plan->debug_stall_role))
        return FD_ERR_INVALID_ARG;
    // the shared memory the plan grants must hold its layout
    {
        fd_problem pk = p;
        pk.B = plan->kv_rows;
        if (plan->scratch_in_stage != 0 && plan->scratch_in_stage != 1) return FD_ERR_INVALID_ARG;
        const size_t need = decode_smem_bytes(pk, ks, plan->stages, plan->scratch_in_stage == 1);
        if (need == 0 || need > (size_t)std::max(0, plan->smem_bytes)) return FD_ERR_INVALID_ARG;
    }

    const int boxr = std::gcd(p.page_size, ks.tile);
    CUtensorMap tmk, tmv;
    if (!encode_pool_map(&tmk, k_pages, p, boxr) || !encode_pool_map(&tmv, v_pages, p, boxr)) return FD_ERR_CUDA;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t rows = (size_t)p.B * p.Hq;
    DecodeParams dp;
    std::memset(&dp, 0, sizeof(dp));
    dp.q = q;
    dp.block_table = block_table;
    dp.seq_lens = seq_lens;
    dp.batch_idx = ex ? ex->cache_batch_idx : nullptr;
    dp.leftpad = ex ? ex->cache_leftpad : nullptr;
    dp.cache_rows = (ex && ex->cache_batch_idx) ? ex->cache_rows : plan->kv_rows;
    dp.k_scale = k_scale;
    dp.v_scale = v_scale;
    dp.out = out;
    dp.lse = lse;
    dp.part_o = reinterpret_cast<float *>(ws + plan->ws_partial_o);
    dp.part_m = reinterpret_cast<float *>(ws + plan->ws_partial_md);
    dp.part_d = dp.part_m + rows * plan->num_splits;
    int *ctr = reinterpret_cast<int *>(ws + plan->ws_counters);
    dp.merge_ctr = ctr;
    dp.work_ctr = ctr + (size_t)plan->kv_rows * p.Hkv * plan->head_subgroups;
    dp.done_ctr = dp.work_ctr + 1;
    dp.status = status_dev;
    dp.B = p.B;
    dp.Hq = p.Hq;
    dp.Hkv = p.Hkv;
    dp.G = p.Hq / p.Hkv;
    dp.fold = fold;
    dp.nhg = plan->head_subgroups;
    dp.Bkv = plan->kv_rows;
    dp.page_size = p.page_size;
    dp.max_blocks = p.max_blocks_per_seq;
    dp.num_pages = p.num_pages;
    dp.S = plan->num_splits;
    dp.chunk = plan->chunk_tokens;
    dp.cap = plan->num_splits * plan->chunk_tokens;
    dp.boxr = boxr;
    dp.out_dtype = p.out_dtype;
    dp.fuse_merge = plan->fuse_merge;
    dp.stages = plan->stages;
    dp.scr_in_stage = plan->scratch_in_stage;
    dp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p.D));
    dp.timeout_ns = plan->timeout_us > 0 ? (uint64_t)plan->timeout_us * 1000ull : kTimeoutNs;
    dp.stall_ns = (uint64_t)plan->debug_stall_us * 1000ull;
    dp.stall_role = plan->debug_stall_role;
    dp.qn = q_len;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_decode(p, ks, dp, tmk, tmv, plan->grid_ctas, (size_t)plan->smem_bytes, s);
    if (e != cudaSuccess) return FD_ERR_CUDA;
    if (!plan->fuse_merge && plan->num_splits > 1) {
        MergeParams mp;
        mp.part_o = dp.part_o;
        mp.part_m = dp.part_m;
        mp.part_d = dp.part_d;
        mp.out = out;
        mp.lse = lse;
        mp.seq_lens = seq_lens;
        mp.batch_idx = dp.batch_idx;
        mp.leftpad = dp.leftpad;
        mp.cache_rows = dp.cache_rows;
        mp.B = p.B;
        mp.Hq = p.Hq;
        mp.S = plan->num_splits;
        mp.D = p.D;
        mp.chunk = plan->chunk_tokens;
        mp.cap = dp.cap;
        mp.fold = fold;
        mp.out_dtype = p.out_dtype;
        e = launch_merge(mp, s);
        if (e != cudaSuccess) return FD_ERR_CUDA;
    }
    return FD_OK;
}

}  // namespace

extern "C" {

fd_status fd_decode_paged(const fd_plan_t *plan, const void *q, const void *k_pages, const void *v_pages,
                          const float *k_scale, const float *v_scale, const int32_t *block_table,
                          const int32_t *seq_lens, void *out, float *lse, void *workspace, size_t workspace_bytes,
                          int32_t *status_dev, void *stream) {
    return decode_impl(plan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, nullptr, out, lse,
                       workspace, workspace_bytes, status_dev, stream);
}

fd_status fd_decode_paged_ex(const fd_plan_t *plan, const void *q, const void *k_pages, const void *v_pages,
                             const float *k_scale, const float *v_scale, const int32_t *block_table,
                             const int32_t *seq_lens, const fd_decode_extras *extras, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream) {
    if (extras) {
        if (extras->cache_batch_idx && extras->cache_rows < 1) return FD_ERR_INVALID_ARG;
        if ((extras->cache_batch_idx && !aligned(extras->cache_batch_idx, 4)) ||
            (extras->cache_leftpad && !aligned(extras->cache_leftpad, 4)))
            return FD_ERR_INVALID_ARG;
    }
    return decode_impl(plan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, extras, out, lse,
                       workspace, workspace_bytes, status_dev, stream);
}

fd_status fd_host_io_layout_for(const fd_plan_t *plan, fd_host_io_layout *layout) {
    if (!plan || !layout) return FD_ERR_INVALID_ARG;
    const fd_problem &p = plan->problem;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rows = (size_t)p.B * p.Hq;
    const size_t kv_rows = (size_t)(plan->kv_rows > 0 ? plan->kv_rows : p.B);
    layout->q_offset = 0;
    layout->block_table_offset = up(rows * p.D * elem_bytes(p.q_dtype));
    layout->seq_lens_offset = layout->block_table_offset + up(kv_rows * p.max_blocks_per_seq * 4);
    layout->in_bytes = layout->seq_lens_offset + up(kv_rows * 4);
    layout->out_offset = 0;
    layout->lse_offset = up(rows * p.D * elem_bytes(p.out_dtype));
    layout->out_bytes = layout->lse_offset + up(rows * 4);
    return FD_OK;
}

fd_status fd_host_copy_in(const fd_plan_t *plan, const void *host_in, void *dev_in, void *stream) {
    if (!plan || !host_in || !dev_in) return FD_ERR_INVALID_ARG;
    if (!aligned(dev_in, 256)) return FD_ERR_INVALID_ARG;
    fd_host_io_layout io;
    fd_host_io_layout_for(plan, &io);
    if (cudaMemcpyAsync(dev_in, host_in, io.in_bytes, cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return FD_ERR_CUDA;
    return FD_OK;
}

fd_status fd_decode_paged_staged(const fd_plan_t *plan, const void *dev_in, const void *k_pages, const void *v_pages,
                                 const float *k_scale, const float *v_scale, void *dev_out, void *host_out,
                                 void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream) {
    if (!plan || !dev_in || !dev_out) return FD_ERR_INVALID_ARG;
    if (!aligned(dev_in, 256) || !aligned(dev_out, 256)) return FD_ERR_INVALID_ARG;
    fd_host_io_layout io;
    fd_host_io_layout_for(plan, &io);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t *in = static_cast<const uint8_t *>(dev_in);
    // When the host output block is page-locked memory mapped for the device
    // (unified addressing), the kernel stores out and lse straight into it:
    // no device-to-host copy follows the decode.
    uint8_t *out = static_cast<uint8_t *>(dev_out);
    bool direct = false;
    cudaPointerAttributes attr;
    if (host_out && cudaPointerGetAttributes(&attr, host_out) == cudaSuccess && attr.type == cudaMemoryTypeHost &&
        attr.devicePointer != nullptr && aligned(attr.devicePointer, 256)) {
        out = static_cast<uint8_t *>(attr.devicePointer);
        direct = true;
    } else if (host_out) {
        cudaGetLastError();  // a pageable pointer is not an error here
    }
    const fd_status r = fd_decode_paged(plan, in + io.q_offset, k_pages, v_pages, k_scale, v_scale,
                                        reinterpret_cast<const int32_t *>(in + io.block_table_offset),
                                        reinterpret_cast<const int32_t *>(in + io.seq_lens_offset),
                                        out + io.out_offset, reinterpret_cast<float *>(out + io.lse_offset),
                                        workspace, workspace_bytes, status_dev, stream);
    if (r != FD_OK) return r;
    if (host_out && !direct &&
        cudaMemcpyAsync(host_out, dev_out, io.out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return FD_ERR_CUDA;
    return FD_OK;
}

fd_status fd_host_copy_out(const fd_plan_t *plan, const void *dev_out, void *host_out, void *stream) {
    if (!plan || !dev_out || !host_out) return FD_ERR_INVALID_ARG;
    if (!aligned(dev_out, 256)) return FD_ERR_INVALID_ARG;
    fd_host_io_layout io;
    fd_host_io_layout_for(plan, &io);
    if (cudaMemcpyAsync(host_out, dev_out, io.out_bytes, cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return FD_ERR_CUDA;
    return FD_OK;
}

fd_status fd_decode_paged_host(const fd_plan_t *plan, const void *host_in, void *dev_in, const void *k_pages,
                               const void *v_pages, const float *k_scale, const float *v_scale, void *dev_out,
                               void *host_out, void *workspace, size_t workspace_bytes, int32_t *status_dev,
                               void *stream) {
    if (!plan || !host_in || !dev_in || !dev_out || !host_out) return FD_ERR_INVALID_ARG;
    if (!aligned(dev_in, 256) || !aligned(dev_out, 256)) return FD_ERR_INVALID_ARG;
    const fd_status r = fd_host_copy_in(plan, host_in, dev_in, stream);
    if (r != FD_OK) return r;
    return fd_decode_paged_staged(plan, dev_in, k_pages, v_pages, k_scale, v_scale, dev_out, host_out, workspace,
                                  workspace_bytes, status_dev, stream);
}

fd_status fd_merge_states(const float *o_part, const float *m, const float *d, int B, int Hq, int S, int D,
                          fd_dtype out_dtype, void *out, float *lse, void *stream) {
    if (!o_part || !m || !d || !out) return FD_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || S < 1 || D < 1) return FD_ERR_INVALID_ARG;
    if (S > 4096 || D > 256) return FD_ERR_UNSUPPORTED;
    if (out_dtype != FD_F16 && out_dtype != FD_BF16 && out_dtype != FD_F32) return FD_ERR_UNSUPPORTED;
    if (!aligned(o_part, 4) || !aligned(m, 4) || !aligned(d, 4) || !aligned(out, elem_bytes(out_dtype)) ||
        (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    MergeParams mp;
    mp.part_o = o_part;
    mp.part_m = m;
    mp.part_d = d;
    mp.out = out;
    mp.lse = lse;
    mp.seq_lens = nullptr;
    mp.batch_idx = nullptr;
    mp.leftpad = nullptr;
    mp.cache_rows = 0;
    mp.B = B;
    mp.Hq = Hq;
    mp.S = S;
    mp.D = D;
    mp.chunk = 1;
    mp.cap = 0;
    mp.fold = 1;
    mp.out_dtype = out_dtype;
    return launch_merge(mp, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

}  // extern "C"

namespace {

fd_status append_impl(const fd_problem *problem, const void *k_new, const void *v_new, void *k_pages,
                      void *v_pages, const float *k_scale, const float *v_scale, const int32_t *block_table,
                      const int32_t *seq_lens, const float *rotary_cos, const float *rotary_sin, int rotary_dim,
                      int max_pos, int interleaved, void *q_inout, int32_t *status_dev, void *stream) {
    fd_status st = validate_problem(problem);
    if (st != FD_OK) return st;
    const fd_problem &p = *problem;
    if (!k_new || !v_new || !k_pages || !v_pages || !block_table || !seq_lens) return FD_ERR_INVALID_ARG;
    const bool fp8 = p.kv_dtype == FD_E4M3;
    if (fp8 != (k_scale != nullptr) || fp8 != (v_scale != nullptr)) return FD_ERR_INVALID_ARG;
    if (!aligned(k_new, 4) || !aligned(v_new, 4) || !aligned(k_pages, 4) || !aligned(v_pages, 4))
        return FD_ERR_INVALID_ARG;
    AppendParams ap;
    ap.k_new = k_new;
    ap.v_new = v_new;
    ap.k_pages = k_pages;
    ap.v_pages = v_pages;
    ap.k_scale = k_scale;
    ap.v_scale = v_scale;
    ap.block_table = block_table;
    ap.seq_lens = seq_lens;
    ap.status = status_dev;
    ap.B = p.B;
    ap.Hkv = p.Hkv;
    ap.D = p.D;
    ap.page_size = p.page_size;
    ap.max_blocks = p.max_blocks_per_seq;
    ap.num_pages = p.num_pages;
    ap.kv_kind = p.kv_dtype == FD_F16 ? KV_F16 : (p.kv_dtype == FD_BF16 ? KV_BF16 : KV_E4M3);
    ap.new_is_bf16 = p.q_dtype == FD_BF16 ? 1 : 0;
    ap.cos = rotary_cos;
    ap.sin = rotary_sin;
    ap.rotary_dim = rotary_dim;
    ap.max_pos = max_pos;
    ap.interleaved = interleaved ? 1 : 0;
    ap.q_inout = q_inout;
    ap.Hq = p.Hq;
    ap.q_is_bf16 = p.q_dtype == FD_BF16 ? 1 : 0;
    return launch_append(ap, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

}  // namespace

extern "C" {

fd_status fd_merge_two(const float *out_a, const float *lse_a, const float *out_b, const float *lse_b, int rows, int D,
                       fd_dtype out_dtype, void *out, float *lse, void *stream) {
    if (!out_a || !lse_a || !out_b || !lse_b || !out || rows < 1 || D < 4 || D % 4) return FD_ERR_INVALID_ARG;
    if (out_dtype != FD_F16 && out_dtype != FD_BF16 && out_dtype != FD_F32) return FD_ERR_UNSUPPORTED;
    if (!aligned(out_a, 16) || !aligned(out_b, 16) || !aligned(lse_a, 4) || !aligned(lse_b, 4) ||
        !aligned(out, elem_bytes(out_dtype)) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    return launch_merge_two(out_a, lse_a, out_b, lse_b, rows, D, out_dtype, out, lse,
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FD_OK
               : FD_ERR_CUDA;
}

fd_status fd_append_kv(const fd_problem *problem, const void *k_new, const void *v_new, void *k_pages,
                       void *v_pages, const float *k_scale, const float *v_scale, const int32_t *block_table,
                       const int32_t *seq_lens, int32_t *status_dev, void *stream) {
    return append_impl(problem, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, nullptr,
                       nullptr, 0, 0, 0, nullptr, status_dev, stream);
}

fd_status fd_append_kv_rotary(const fd_problem *problem, const void *k_new, const void *v_new, void *k_pages,
                              void *v_pages, const float *k_scale, const float *v_scale,
                              const int32_t *block_table, const int32_t *seq_lens, const float *rotary_cos,
                              const float *rotary_sin, int rotary_dim, int max_pos, int interleaved, void *q_inout,
                              int32_t *status_dev, void *stream) {
    if (!problem || !rotary_cos || !rotary_sin || max_pos < 1 || rotary_dim < 2 || (rotary_dim & 1) ||
        rotary_dim > problem->D || !aligned(rotary_cos, 4) || !aligned(rotary_sin, 4) ||
        (q_inout && !aligned(q_inout, 4)))
        return FD_ERR_INVALID_ARG;
    return append_impl(problem, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, rotary_cos,
                       rotary_sin, rotary_dim, max_pos, interleaved, q_inout, status_dev, stream);
}

}  // extern "C"

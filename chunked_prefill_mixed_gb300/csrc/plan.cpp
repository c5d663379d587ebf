// plan.cpp -- host planner of libsarathi: the stall-free budgeted batch, its
// ragged-batch metadata and the step kernel's work list.
//
// Budget order follows "Chunked Prefill 与 PD 分离" §3.1 (running decodes, then
// unfinished prefill chunks, then new requests) and the per-request chunk of
// "分块预填充与 Stall-free 调度" §六·补二 (min of the budget left and the prompt
// left).  Several prefills may share one budget, "Sarathi-Serve 完全拆解"
// §"一个 512-token 预算的例子".  Metadata arrays as named in "Sarathi-Serve 完全拆解"
// §"混合批不是把两类注意力强行做成同一个形状".
#include <algorithm>
#include <array>
#include <cstdio>
#include <cstring>
#include <functional>
#include <string>
#include <vector>

#include "sarathi.h"
#include "sarathi_internal.h"

namespace sarathi {

static thread_local std::string g_last_error = "";

void set_error(const char* msg) { g_last_error = msg ? msg : ""; }

int32_t fail(int32_t code, const char* msg) {
    set_error(msg);
    return code;
}

int32_t check_shape(const sarathi_shape* sh) {
    if (!sh) return fail(SARATHI_ERR_INVALID_ARG, "shape is NULL");
    if (sh->num_heads_q <= 0 || sh->num_heads_kv <= 0 || sh->head_dim <= 0 || sh->page_size <= 0)
        return fail(SARATHI_ERR_INVALID_ARG, "shape fields must be positive");
    if (sh->num_heads_q % sh->num_heads_kv != 0)
        return fail(SARATHI_ERR_INVALID_ARG, "num_heads_q must be a multiple of num_heads_kv");
    if (sh->page_size != kPage) return fail(SARATHI_ERR_UNSUPPORTED, "page_size must be 16");
    if (sh->head_dim != 64 && sh->head_dim != 128)
        return fail(SARATHI_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (sh->num_heads_q / sh->num_heads_kv > kMaxGroup)
        return fail(SARATHI_ERR_UNSUPPORTED, "q heads per kv head must be <= 16");
    return SARATHI_OK;
}

namespace {

struct Sched {
    int32_t req;
    int32_t n;
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int32_t validate_requests(const sarathi_request* reqs, int32_t n_reqs) {
    if (n_reqs < 0) return fail(SARATHI_ERR_INVALID_ARG, "n_reqs < 0");
    if (n_reqs > 0 && !reqs) return fail(SARATHI_ERR_INVALID_ARG, "reqs is NULL");
    for (int32_t i = 0; i < n_reqs; ++i) {
        const sarathi_request& r = reqs[i];
        if (r.state < SARATHI_DECODE || r.state > SARATHI_PREFILL_WAITING)
            return fail(SARATHI_ERR_INVALID_ARG, "request state out of range");
        if (r.num_computed < 0) return fail(SARATHI_ERR_INVALID_ARG, "num_computed < 0");
        if (r.state != SARATHI_DECODE && r.prompt_len < r.num_computed)
            return fail(SARATHI_ERR_INVALID_ARG, "prefill with num_computed > prompt_len");
        if (r.num_pages < 0 || (r.num_pages > 0 && !r.pages))
            return fail(SARATHI_ERR_INVALID_ARG, "bad block table");
    }
    return SARATHI_OK;
}

// Cost model that orders the work list (longest first) and sizes the SM
// partition between its two queues, fitted to per-item times of the step
// kernel on GB300 and to step times over the partition size: a prefill tile
// costs a fixed start (Q fill, first loads, epilogue) plus its 128-key blocks
// at tensor-core speed; a decode split a fixed start plus its pages at an
// equal share of HBM bandwidth (every SM streaming), or at one SM's own rate
// while fewer SMs stream than saturate HBM.
constexpr double kPrefillFixedNs = 6500.0;
constexpr double kPrefillFlopPerNs = 9000.0;
constexpr double kDecodeFixedNs = 2000.0;
constexpr double kDecodeBytesPerNs = 40.0;       // a decode split's share of HBM with every SM streaming
constexpr double kDecodeAloneBytesPerNs = 80.0;  // one SM's own streaming rate when HBM has room
constexpr double kHbmBytesPerNs = 6500.0;        // the whole GPU
// an APPEND item: per (token, kv head) it rotates and stores
constexpr double kAppendFixedNs = 1500.0;
constexpr double kAppendNsPerTokenHead = 45.0;
// a key piece of a split tile: a tile's fixed start, plus its partial's
// write, the merge (by the last piece) and the slower blocks of pieces that
// share fewer pages with the tiles running beside them (fitted to step times
// of prefill-only steps cut at 512, 1024 and 2048 tokens)
constexpr double kPieceExtraNs = 8000.0;
// The simulation of a step without decodes has a fit of its own, to item
// times (per-CTA timelines) and step times of prefill-only steps on GB300 --
// chunks of 512, 1024 and 2048 tokens after 6144-7680 tokens of history, the
// APPEND items on the one queue or beside the tiles, with and without key
// pieces: a 128-key block of a tile (d = 128; in proportion to d), the
// tile's start before its first block and its end after the last, the
// APPEND item's time as a factor of its estimate above when every CTA
// appends at the start of the step (A) and when a few append beside the
// tiles (B), and the extra cost of a key piece.
constexpr double kSoloBlockNs = 790.0;
constexpr double kSoloPreNs = 4000.0;
constexpr double kSoloPostNs = 3000.0;
constexpr double kSoloAppendA = 1.09;
constexpr double kSoloAppendB = 0.92;
constexpr double kSoloPieceExtraNs = 5000.0;

}  // namespace
}  // namespace sarathi

using namespace sarathi;

extern "C" const char* sarathi_last_error(void) { return g_last_error.c_str(); }

extern "C" int32_t sarathi_abi_version(void) { return SARATHI_ABI_VERSION; }

extern "C" int32_t sarathi_plan_bounds(const sarathi_request* reqs, int32_t n_reqs, int32_t token_budget,
                                       const sarathi_shape* shape, int32_t num_sms,
                                       size_t* host_buf_bytes, size_t* device_workspace_bytes) {
    int32_t st = check_shape(shape);
    if (st) return st;
    st = validate_requests(reqs, n_reqs);
    if (st) return st;
    if (token_budget <= 0) return fail(SARATHI_ERR_INVALID_ARG, "token_budget must be positive");
    if (num_sms <= 0) return fail(SARATHI_ERR_INVALID_ARG, "num_sms must be positive");
    const int64_t Hkv = shape->num_heads_kv;
    const int group = shape->num_heads_q / shape->num_heads_kv;
    int64_t n_dec = 0, pages = 0;
    for (int32_t i = 0; i < n_reqs; ++i) {
        n_dec += reqs[i].state == SARATHI_DECODE;
        pages += reqs[i].num_pages;
    }
    const int64_t n = n_reqs;
    const int64_t T = n_dec + token_budget;
    // APPEND items: each row's tokens cut where their positions cross a
    // 128-position boundary, times the groups of kv heads
    const int64_t appends = (T / kTileRows + 2 * n) * kv_groups((int)Hkv);
    const int64_t tiles = (T / tokens_per_tile(group) + n) * Hkv;
    // decode splits: sum over one-token rows (decodes, and prefill chunks of one
    // token) and kv heads of ceil(np / split) with split >= their page-heads /
    // (num_sms * kDecodeItemsPerSm), so at most num_sms * kDecodeItemsPerSm +
    // (rows x kv heads) items
    const int64_t dec_items =
        std::min<int64_t>((pages / kDecodeMinSplitPages + n) * Hkv, (int64_t)num_sms * kDecodeItemsPerSm + n * Hkv);
    // key pieces: at most num_sms tiles of a step are split, into at most
    // kMaxPieces pieces each
    const int64_t pieces_extra = (int64_t)num_sms * (kMaxPieces - 1);
    const int64_t items = appends + tiles + dec_items + pieces_extra;
    const int64_t ints = 6 * n + 2 + pages + 8 + items * kItemInts;
    if (host_buf_bytes) *host_buf_bytes = (size_t)ints * 4;
    if (device_workspace_bytes) {
        const int64_t n_merge = n * Hkv + num_sms;
        const int64_t slots = dec_items + 1 + (int64_t)num_sms * kMaxPieces * pf_piece_slots(group);
        *device_workspace_bytes = (size_t)(partial_offset_bytes((int)n, (int)n_merge, (int)T, (int)Hkv) +
                                           slots * partial_slot_floats(group, shape->head_dim) * 4);
    }
    return SARATHI_OK;
}

// A chunk that does not finish its prompt is cut down to a multiple of align
// ("Sarathi-Serve 完全拆解", §"257 为什么可能比 256 慢 32%"); a prompt's final
// chunk keeps its size.
inline int64_t aligned_take(int64_t take, int64_t rem, int32_t align) {
    return (align > 1 && take < rem) ? take - take % align : take;
}

extern "C" int32_t sarathi_plan(const sarathi_request* reqs, int32_t n_reqs, int32_t token_budget,
                                const sarathi_shape* shape, int32_t num_sms,
                                int32_t* host_buf, size_t host_buf_bytes, sarathi_plan_info* info) {
    const sarathi_plan_policy policy = {SARATHI_POLICY_STALL_FREE, token_budget, 0, 1};
    return sarathi_plan_ex(reqs, n_reqs, &policy, shape, num_sms, host_buf, host_buf_bytes, info);
}

namespace {
// The head of a work item (fields kKind..kNSplit); the rest is filled when the
// item is written into the packed plan.
using ItemHead = std::array<int32_t, 8>;
struct Timed {
    double ns_est;
    ItemHead it;
};
// Per-thread buffers reused across calls: a step's plan allocates nothing once
// the buffers have grown to its size.
struct PlanScratch {
    std::vector<Sched> sched;
    std::vector<int32_t> np, hist, aux;
    std::vector<ItemHead> appends;
    std::vector<Timed> tiles, decs;
    std::vector<double> key, pred, heap, snaps, flag, flag_pm;
    std::vector<int64_t> grp;
    std::vector<uint32_t> pf_order, dec_order, bucket;
};
thread_local PlanScratch t_scratch;
}  // namespace

extern "C" int32_t sarathi_plan_ex(const sarathi_request* reqs, int32_t n_reqs, const sarathi_plan_policy* policy,
                                   const sarathi_shape* shape, int32_t num_sms,
                                   int32_t* host_buf, size_t host_buf_bytes, sarathi_plan_info* info) {
    if (!info) return fail(SARATHI_ERR_INVALID_ARG, "info is NULL");
    std::memset(info, 0, sizeof *info);
    if (!policy) return fail(SARATHI_ERR_INVALID_ARG, "policy is NULL");
    int32_t st = check_shape(shape);
    if (st) return st;
    st = validate_requests(reqs, n_reqs);
    if (st) return st;
    const int32_t token_budget = policy->token_budget;
    if (policy->kind != SARATHI_POLICY_STALL_FREE && policy->kind != SARATHI_POLICY_DECODE_MAXIMAL)
        return fail(SARATHI_ERR_INVALID_ARG, "unknown policy kind");
    if (token_budget <= 0) return fail(SARATHI_ERR_INVALID_ARG, "token_budget must be positive");
    if (policy->chunk_align < 1) return fail(SARATHI_ERR_INVALID_ARG, "chunk_align must be >= 1");
    if (policy->max_batch < 0 || (policy->kind == SARATHI_POLICY_STALL_FREE && policy->max_batch != 0))
        return fail(SARATHI_ERR_INVALID_ARG, "max_batch must be 0 (stall-free) or >= 0 (decode-maximal)");
    if (num_sms <= 0) return fail(SARATHI_ERR_INVALID_ARG, "num_sms must be positive");

    const int Hkv = shape->num_heads_kv;
    const int group = shape->num_heads_q / Hkv;
    const int d = shape->head_dim;

    PlanScratch& sc = t_scratch;
    // ---- 1. the batch
    std::vector<Sched>& sched = sc.sched;
    sched.clear();
    int32_t decodes = 0;
    const int32_t align = policy->chunk_align;
    if (policy->kind == SARATHI_POLICY_STALL_FREE) {
        // decodes, running prefills, waiting prefills, each chunk as large as
        // the budget left allows
        int64_t left = token_budget;
        for (int32_t i = 0; i < n_reqs; ++i)
            if (reqs[i].state == SARATHI_DECODE) {
                sched.push_back({i, 1});
                ++decodes;
                --left;
            }
        for (int cls = SARATHI_PREFILL_RUNNING; cls <= SARATHI_PREFILL_WAITING; ++cls)
            for (int32_t i = 0; i < n_reqs; ++i) {
                if (reqs[i].state != cls) continue;
                int64_t rem = (int64_t)reqs[i].prompt_len - reqs[i].num_computed;
                int64_t take = aligned_take(std::min<int64_t>(rem, std::max<int64_t>(left, 0)), rem, align);
                if (take <= 0) continue;
                sched.push_back({i, (int32_t)take});
                left -= take;
            }
    } else {
        // decode-maximal ("Sarathi：让解码搭上 prefill 的顺风车", §"Decode-maximal
        // batching：顺车的账本"): one chunk, then up to B - 1 decodes beside it
        int32_t chunk_req = -1;
        int64_t chunk_take = 0;
        for (int cls = SARATHI_PREFILL_RUNNING; cls <= SARATHI_PREFILL_WAITING && chunk_req < 0; ++cls)
            for (int32_t i = 0; i < n_reqs; ++i) {
                if (reqs[i].state != cls) continue;
                int64_t rem = (int64_t)reqs[i].prompt_len - reqs[i].num_computed;
                if (rem <= 0) continue;
                chunk_req = i;
                chunk_take = aligned_take(std::min<int64_t>(rem, token_budget), rem, align);
                break;
            }
        if (chunk_take <= 0) chunk_req = -1;
        const int64_t cap =
            policy->max_batch > 0 ? (int64_t)policy->max_batch - (chunk_req >= 0 ? 1 : 0) : (int64_t)n_reqs;
        for (int32_t i = 0; i < n_reqs && decodes < cap; ++i)
            if (reqs[i].state == SARATHI_DECODE) {
                sched.push_back({i, 1});
                ++decodes;
            }
        if (chunk_req >= 0) sched.push_back({chunk_req, (int32_t)chunk_take});
    }
    const int32_t ns = (int32_t)sched.size();

    // ---- 2. per-row KV extent, checked against the block tables
    std::vector<int32_t>& np = sc.np;
    std::vector<int32_t>& hist = sc.hist;
    np.assign(ns, 0);
    hist.assign(ns, 0);
    int64_t nnz = 0, T = 0, pairs = 0, history = 0;
    int32_t max_kv = 0;
    for (int32_t s = 0; s < ns; ++s) {
        const sarathi_request& r = reqs[sched[s].req];
        int64_t kv_len = (int64_t)r.num_computed + sched[s].n;
        int64_t p = ceil_div(kv_len, kPage);
        if (p > r.num_pages) {
            char msg[160];
            std::snprintf(msg, sizeof msg, "request %d needs %lld pages, block table has %d", sched[s].req,
                          (long long)p, r.num_pages);
            return fail(SARATHI_ERR_CAPACITY, msg);
        }
        np[s] = (int32_t)p;
        hist[s] = r.num_computed;
        nnz += p;
        T += sched[s].n;
        const int64_t n = sched[s].n, h = r.num_computed;
        pairs += n * h + n * (n + 1) / 2;
        history += h;
        max_kv = std::max<int32_t>(max_kv, (int32_t)kv_len);
    }

    // ---- 3. work list
    std::vector<int32_t>& aux = sc.aux;
    aux.assign(ns, 0);
    std::vector<ItemHead>& appends = sc.appends;
    std::vector<Timed>& tiles = sc.tiles;
    std::vector<Timed>& decs = sc.decs;
    appends.clear();
    tiles.clear();
    decs.clear();
    const int tpt = tokens_per_tile(group);
    const int tpi = tokens_per_item(group);
    // decode split size from the total decode pages and the SM count
    int64_t dec_page_heads = 0;
    for (int32_t s = 0; s < ns; ++s)
        if (sched[s].n == 1) dec_page_heads += (int64_t)np[s] * Hkv;
    const int64_t target = (int64_t)num_sms * kDecodeItemsPerSm;
    const int64_t split =
        std::max<int64_t>(kDecodeMinSplitPages, ceil_div(std::max<int64_t>(dec_page_heads, 1), target));
    int32_t n_partials = 0, n_merge = 0, n_flags = 0;
    const double kv_page_bytes = 2.0 * kPage * d * 2;
    for (int32_t s = 0; s < ns; ++s) {
        const int32_t n = sched[s].n;
        const int32_t h = hist[s];
        if (n >= 2) {
            // prefill-like: append items first (the row's tokens cut where their
            // positions cross a 128-position boundary -- a K/V block of the
            // tiles -- times the groups of kv heads; each sets one ready flag,
            // the row's flags from aux[s] on), then one tile per (kv head,
            // token block)
            aux[s] = n_flags;
            for (int32_t t0 = 0; t0 < n;) {
                const int32_t c = std::min<int32_t>(n - t0, kTileRows - (h + t0) % kTileRows);
                for (int g0 = 0; g0 < Hkv; g0 += kAppendHeads) {
                    appends.push_back({kAppend, s, g0, t0, c, -1, -1, 0});
                    ++n_flags;
                }
                t0 += c;
            }
            // one (request, kv head) at a time, costliest item first: the items
            // that read the same history pages run side by side and share L2
            for (int g = 0; g < Hkv; ++g)
                for (int32_t t0 = (n - 1) / tpi * tpi; t0 >= 0; t0 -= tpi) {
                    int32_t c = std::min(tpi, n - t0);
                    const double keys = (double)ceil_div((int64_t)h + t0 + c, kTileRows) * kTileRows;
                    const double flops = 4.0 * d * kTileRows * ceil_div(c, tpt) * keys;
                    tiles.push_back(
                        {kPrefillFixedNs + flops / kPrefillFlopPerNs, {kPrefill, s, g, t0, c, -1, -1, 0}});
                }
        } else {
            // decode-like: split the pages; an item covers up to kDecodeHeads kv
            // heads (sharing its start-up over them); the item holding the last
            // page also appends the new token's K/V for its heads.
            // (nsplit-1)*per < np always holds, so no split is empty.
            const int64_t nsplit = ceil_div(np[s], split);
            const int64_t per = ceil_div(np[s], nsplit);
            for (int g = 0; g < Hkv; g += kDecodeHeads) {
                const int ngh = std::min(kDecodeHeads, Hkv - g);
                int32_t merge = nsplit > 1 ? n_merge++ : -1;
                int32_t first = nsplit > 1 ? n_partials : -1;
                if (nsplit > 1) n_partials += (int32_t)(nsplit * ngh);
                for (int64_t k = 0; k < nsplit; ++k) {
                    int32_t p0 = (int32_t)(k * per);
                    int32_t pc = (int32_t)std::min<int64_t>(per, np[s] - p0);
                    decs.push_back({kDecodeFixedNs + pc * ngh * kv_page_bytes / kDecodeBytesPerNs,
                                    {kDecode, s, g, p0, pc, first, merge, (int32_t)nsplit}});
                }
            }
        }
    }
    // Two queues.  The first holds the prefill tiles, longest first (the tiles
    // of one (request, kv head) read the same pages, so they stay contiguous:
    // the group sorts by its costliest tile); the second the decode splits,
    // longest first.  CTAs [0, first_sms) take items from the first queue and
    // the others from the second, each falling back to the other queue once its
    // own is empty: the compute-bound prefill tiles run on a partition of the
    // SMs for the whole step while the other SMs stream the decodes' KV at the
    // full HBM rate (with every SM on prefill at the start of a step, the
    // decodes would stream from a few SMs meanwhile); first_sms comes from a
    // fluid model of the two sides (below).  APPEND items lead
    // the second queue (they never wait, so the streaming CTAs take them first
    // and the tiles that wait for them are not held up); in a step without
    // decodes they lead the one queue, or make up the second (3b).  (The sorts move 4-byte indices, not the items.)
    const size_t n_tiles = tiles.size();
    std::vector<double>& key = sc.key;
    std::vector<int64_t>& grp = sc.grp;
    key.resize(n_tiles);
    grp.resize(n_tiles);
    for (size_t i = 0; i < n_tiles;) {
        size_t e = i;
        const int32_t s0 = tiles[i].it[kS], g0 = tiles[i].it[kG];
        double mx = 0;
        while (e < n_tiles && tiles[e].it[kS] == s0 && tiles[e].it[kG] == g0) mx = std::max(mx, tiles[e++].ns_est);
        for (; i < e; ++i) {
            key[i] = mx;
            grp[i] = (int64_t)s0 * Hkv + g0;
        }
    }
    std::vector<uint32_t>& pf_order = sc.pf_order;
    std::vector<uint32_t>& dec_order = sc.dec_order;
    pf_order.resize(n_tiles);
    dec_order.resize(decs.size());
    for (size_t i = 0; i < n_tiles; ++i) pf_order[i] = (uint32_t)i;
    std::stable_sort(pf_order.begin(), pf_order.end(), [&](uint32_t a, uint32_t b) {
        if (key[a] != key[b]) return key[a] > key[b];
        return grp[a] < grp[b];
    });
    {
        // a decode split's estimate grows with its page count: a stable
        // counting sort on the count, largest first
        int32_t max_pc = 0;
        for (auto& t : decs) max_pc = std::max(max_pc, t.it[kCount]);
        std::vector<uint32_t>& bucket = sc.bucket;
        bucket.assign((size_t)max_pc + 2, 0);
        for (auto& t : decs) ++bucket[(size_t)(max_pc - t.it[kCount]) + 1];
        for (size_t c = 1; c < bucket.size(); ++c) bucket[c] += bucket[c - 1];
        for (size_t i = 0; i < decs.size(); ++i) dec_order[bucket[(size_t)(max_pc - decs[i].it[kCount])]++] = (uint32_t)i;
    }
    int32_t first_sms = 0;
    if (!tiles.empty() && decs.empty()) {
        first_sms = num_sms;
    } else if (!tiles.empty() && num_sms > 1) {
        double wp = 0, maxp = 0, dec_bytes = 0;
        for (auto& t : tiles) {
            wp += t.ns_est;
            maxp = std::max(maxp, t.ns_est);
        }
        for (auto& t : decs) dec_bytes += t.it[kCount] * std::min(kDecodeHeads, Hkv - t.it[kG]) * kv_page_bytes;
        // Fluid model of the step with k CTAs on the first queue (more than
        // n_tiles act as n_tiles: the rest find it empty and move on): the
        // tiles take wp / k; the decodes stream from the other SMs at
        // min(SMs x one SM's rate, HBM rate); whichever side ends first hands
        // its SMs to the other.  The predicted step is flat over a range of k
        // (the decode streams saturate HBM and the tiles end in time); take
        // the middle of the range within 0.5% of the minimum, away from both
        // edges where the model's error costs most.
        const double r_all = std::min(num_sms * kDecodeAloneBytesPerNs, kHbmBytesPerNs);
        std::vector<double>& pred = sc.pred;
        pred.assign(num_sms, 0.0);
        double best = 0;
        for (int32_t k = 1; k < num_sms; ++k) {
            const double ke = (double)std::min<size_t>((size_t)k, n_tiles);
            const double r1 = std::min((num_sms - ke) * kDecodeAloneBytesPerNs, kHbmBytesPerNs);
            const double tp = wp / ke, td = dec_bytes / r1;
            double t = tp <= td ? tp + (dec_bytes - tp * r1) / r_all : td + (wp - ke * td) / num_sms;
            pred[k] = t = std::max(t, maxp);
            if (k == 1 || t < best) best = t;
        }
        int32_t lo = 0, hi = 0;
        for (int32_t k = 1; k < num_sms; ++k)
            if (pred[k] <= best * 1.005) {
                if (!lo) lo = k;
                hi = k;
            }
        first_sms = std::min<int32_t>((lo + hi) / 2, (int32_t)n_tiles);
    }
    // ---- 3b. prefill-only steps (no decodes): where the APPEND items run, and
    // key pieces for the last tiles.  Two layouts are simulated with the cost
    // model.  (A) One queue, the APPEND items first: every CTA appends, then
    // takes tiles.  (B) The tiles on the first queue and the APPEND items on the
    // second, which app_sms CTAs start on (they never wait, so the tiles that
    // wait for a ready flag are not held up): the tiles stream their history
    // blocks while the chunk's new K/V is appended beside them, and wait only
    // if they reach a chunk block before its APPEND item is done.  Either way
    // the APPEND items never wait, so they are list-scheduled first on the CTAs
    // that take them, and their ends are the ready-flag times; the tiles then
    // start on the CTA that frees first and wait at each chunk block for its
    // flag.  Tiles of similar cost leave a last wave that can hold a few SMs
    // busy while the rest idle; cutting the last split_k tiles into split_n
    // pieces along their 128-key blocks (merged by log-sum-exp, like decode
    // splits) trades a fixed cost per piece for a finer tail (in layout A
    // only).  Layout B is kept only where the model gains clearly over A.
    bool apps_first = decs.empty();
    int32_t app_sms = 0;
    int64_t split_k = 0;
    int32_t split_n = 1;
    auto tile_blocks = [&](const ItemHead& t) {
        return (int32_t)ceil_div((int64_t)hist[t[kS]] + t[kStart] + t[kCount], kTileRows);
    };
    if (decs.empty() && n_tiles >= 1 && num_sms > 1) {
        std::vector<double>& heap = sc.heap;
        std::vector<double>& snaps = sc.snaps;
        std::vector<double>& flag = sc.flag;
        std::vector<double>& flag_pm = sc.flag_pm;
        flag.resize(appends.size());
        flag_pm.resize(appends.size());
        // every tile block costs the same (an M = 128 tile of 128 keys)
        const double blk = kSoloBlockNs * d / 128.0;
        // a min-heap of the CTAs' free times: the CTA that frees first takes
        // the next item.  Its new free time replaces the top: the hole moves
        // down along the smaller children to a leaf (a fixed trip count, no
        // data-dependent branch but the child pick), then the new time rises
        // to its place -- a step or two, as it is usually among the latest.
        auto replace_top = [&](double e) {
            const size_t n = heap.size();
            double* h = heap.data();
            size_t i = 0;
            for (size_t c = 1; c < n; c = 2 * i + 1) {
                c += (c + 1 < n) & (h[c + 1 < n ? c + 1 : c] < h[c]);
                h[i] = h[c];
                i = c;
            }
            while (i > 0) {
                const size_t q = (i - 1) / 2;
                if (h[q] <= e) break;
                h[i] = h[q];
                i = q;
            }
            h[i] = e;
            return e;
        };
        // the end of a tile's key blocks [b0, b1) started at t: block j of the
        // chunk's own keys (j >= jc) starts once the one before has ended and
        // its flag f_j is set, so the blocks end at
        // max(t_jc + (b1 - jc) blk, max_j (f_j + (b1 - j) blk)), t_jc the end of
        // the history blocks.  flag_pm holds the running max of f_j - j blk
        // over a (row, kv-head group)'s blocks, for whole tiles (b0 = 0).
        const int32_t fs = kv_groups(Hkv);
        auto tile_end = [&](const Timed& t, int32_t b0, int32_t b1, double start, double extra) {
            const int32_t s = t.it[kS];
            const int32_t jc = hist[s] / kTileRows;
            double e = start + kSoloPreNs + blk * std::max(0, std::min(b1, jc) - b0);
            const int64_t f0 = aux[s] + t.it[kG] / kAppendHeads - (int64_t)jc * fs;
            if (b0 == 0 && b1 > jc)
                e = std::max(e + blk * (b1 - jc), flag_pm[f0 + (int64_t)(b1 - 1) * fs] + blk * b1);
            else
                for (int32_t j = std::max(b0, jc); j < b1; ++j) e = std::max(e, flag[f0 + (int64_t)j * fs]) + blk;
            return e + kSoloPostNs + extra;
        };
        // candidate split_k: a quarter and a half of the SM count (more
        // measured no better)
        constexpr int kCand = 2;
        int64_t cand[kCand];
        int n_cand = 0;
        for (int q = 1; q <= kCand; ++q) {
            const int64_t k = std::min<int64_t>((int64_t)num_sms * q / 4, (int64_t)n_tiles);
            if (k > 0 && (n_cand == 0 || k != cand[n_cand - 1])) cand[n_cand++] = k;
        }
        // one layout (k APPEND CTAs, 0 = layout A); with_pieces also searches
        // the tail split.  Returns the step's predicted end.
        auto simulate = [&](int32_t k, bool with_pieces, int64_t* sk, int32_t* sn) {
            heap.assign((size_t)(k > 0 ? k : num_sms), 0.0);
            for (size_t i = 0; i < appends.size(); ++i) {
                const ItemHead& a = appends[i];
                flag[i] = replace_top(heap[0] + (k > 0 ? kSoloAppendB : kSoloAppendA) *
                                                    (kAppendFixedNs + kAppendNsPerTokenHead * a[kCount] *
                                                                          std::min<int>(kAppendHeads, Hkv - a[kG])));
            }
            for (int32_t s = 0; s < ns; ++s) {
                if (sched[s].n < 2) continue;
                const int32_t jc = hist[s] / kTileRows;
                const int32_t nbk = (int32_t)ceil_div((int64_t)hist[s] + sched[s].n, kTileRows) - jc;
                for (int32_t gg = 0; gg < fs; ++gg) {
                    double m = -1e300;
                    for (int32_t j = 0; j < nbk; ++j) {
                        const int64_t i = aux[s] + (int64_t)j * fs + gg;
                        m = std::max(m, flag[i] - blk * (jc + j));
                        flag_pm[i] = m;
                    }
                }
            }
            heap.resize((size_t)num_sms, 0.0);
            std::make_heap(heap.begin(), heap.end(), std::greater<double>());
            if (with_pieces) snaps.resize((size_t)n_cand * num_sms);
            for (size_t i = 0; i < n_tiles; ++i) {
                if (with_pieces)
                    for (int c = 0; c < n_cand; ++c)
                        if ((int64_t)(n_tiles - i) == cand[c])
                            std::copy(heap.begin(), heap.end(), snaps.begin() + (size_t)c * num_sms);
                const Timed& t = tiles[pf_order[i]];
                replace_top(tile_end(t, 0, tile_blocks(t.it), heap[0], 0.0));
            }
            double best = *std::max_element(heap.begin(), heap.end());
            *sk = 0;
            *sn = 1;
            if (!with_pieces) return best;
            const double unsplit = best;
            for (int c = 0; c < n_cand; ++c) {
                for (int32_t n = 2; n <= kMaxPieces; ++n) {
                    heap.assign(snaps.begin() + (size_t)c * num_sms, snaps.begin() + (size_t)(c + 1) * num_sms);
                    double m = *std::max_element(heap.begin(), heap.end());
                    for (size_t i = n_tiles - (size_t)cand[c]; i < n_tiles && m < best; ++i) {
                        const Timed& t = tiles[pf_order[i]];
                        const int32_t nb = tile_blocks(t.it);
                        if (nb < 2 * n) {
                            m = std::max(m, replace_top(tile_end(t, 0, nb, heap[0], 0.0)));
                            continue;
                        }
                        for (int32_t q = 0; q < n; ++q)
                            m = std::max(m, replace_top(tile_end(t, (int32_t)((int64_t)nb * q / n),
                                                                 (int32_t)((int64_t)nb * (q + 1) / n), heap[0],
                                                                 kSoloPieceExtraNs)));
                    }
                    if (m < best) {
                        best = m;
                        *sk = cand[c];
                        *sn = n;
                    }
                }
            }
            // keep the plain schedule unless the model gains clearly
            if (best > unsplit * 0.97) {
                *sk = 0;
                *sn = 1;
                return unsplit;
            }
            return best;
        };
        const double t_a = simulate(0, n_tiles >= 2, &split_k, &split_n);
        // layout B can only gain where some tile streams history for longer
        // than an APPEND item takes before it needs a ready flag
        int32_t max_jc = 0;
        for (int32_t s = 0; s < ns; ++s)
            if (sched[s].n >= 2) max_jc = std::max(max_jc, hist[s] / kTileRows);
        const double app_full = kAppendFixedNs + kAppendNsPerTokenHead * kTileRows * std::min(kAppendHeads, Hkv);
        if (!appends.empty() && n_tiles >= 2 && kSoloPreNs + max_jc * blk > kSoloAppendB * app_full) {
            // layout B's candidates: the CTAs left over by w full waves of
            // tiles, a quarter and a half of the SMs; at most half the SMs and
            // at most one CTA per APPEND item
            const int64_t kmax = std::min<int64_t>(num_sms / 2, (int64_t)appends.size());
            int32_t kc[6];
            int n_kc = 0;
            auto add = [&](int64_t k) {
                k = std::max<int64_t>(k, (int64_t)num_sms - (int64_t)n_tiles);  // tile CTAs <= tiles
                if (k < 1 || k > kmax) return;
                for (int i = 0; i < n_kc; ++i)
                    if (kc[i] == k) return;
                kc[n_kc++] = (int32_t)k;
            };
            for (int64_t w = 1; w <= 4; ++w) add((int64_t)num_sms - ceil_div((int64_t)n_tiles, w));
            add(num_sms / 4);
            add(num_sms / 2);
            int64_t sk;
            int32_t sn;
            double t_b = 0;
            int32_t k_b = 0;
            for (int i = 0; i < n_kc; ++i) {
                const double t = simulate(kc[i], false, &sk, &sn);
                if (!k_b || t < t_b) {
                    t_b = t;
                    k_b = kc[i];
                }
            }
            // layout B runs without key pieces: with the APPEND items beside
            // the tiles, pieces measured slower than the plain tail
            if (k_b && t_b < t_a * 0.98) {
                app_sms = k_b;
                apps_first = false;
                split_k = 0;
                split_n = 1;
            }
        }
    }
    if (app_sms > 0) first_sms = num_sms - app_sms;
    int64_t n_pieces_extra = 0;
    for (size_t i = n_tiles - (size_t)split_k; i < n_tiles; ++i)
        if (tile_blocks(tiles[pf_order[i]].it) >= 2 * split_n) n_pieces_extra += split_n - 1;
    const int64_t n_first = (int64_t)n_tiles + n_pieces_extra + (apps_first ? (int64_t)appends.size() : 0);
    const int64_t n_items = (int64_t)n_tiles + n_pieces_extra + (int64_t)appends.size() + (int64_t)decs.size();
    // partial slots and merge groups of the pieces (after the decodes')
    int32_t piece_slot0 = n_partials + ((group & 1) && (n_partials & 1) ? 1 : 0);
    const int32_t piece_merge0 = n_merge;
    const int32_t n_split_tiles = (int32_t)(n_pieces_extra / std::max(split_n - 1, 1));
    if (n_split_tiles > 0) {
        n_partials = piece_slot0 + n_split_tiles * split_n * pf_piece_slots(group);
        n_merge += n_split_tiles;
    }

    // ---- 4. packed layout
    int64_t off = 0;
    auto take = [&](int64_t count) {
        int64_t o = off;
        off += count;
        return (int32_t)o;
    };
    info->off_req_index = take(ns);
    info->off_num_new = take(ns);
    info->off_last_chunk = take(ns);
    info->off_qo_indptr = take(ns + 1);
    info->off_kv_page_indptr = take(ns + 1);
    info->off_kv_page_indices = take(nnz);
    info->off_kv_last_page_len = take(ns);
    info->off_req_aux = take(ns);
    off = (off + 3) / 4 * 4;  // items start on a 16-byte boundary
    info->off_items = take(n_items * kItemInts);
    info->packed_ints = (int32_t)off;
    info->n_sched = ns;
    info->num_decodes = decodes;
    info->num_tokens = (int32_t)T;
    info->nnz_pages = (int32_t)nnz;
    info->n_items = (int32_t)n_items;
    info->n_partials = n_partials;
    info->n_merge = n_merge;
    info->n_first = (int32_t)n_first;
    info->first_sms = n_first == 0 ? 0 : (n_first == n_items ? num_sms : first_sms);
    info->max_kv_len = max_kv;
    info->pairs = pairs;
    info->history_tokens = history;
    info->workspace_bytes =
        partial_offset_bytes(ns, n_merge, (int)T, Hkv) + (int64_t)n_partials * partial_slot_floats(group, d) * 4;
    if (!host_buf || host_buf_bytes < (size_t)off * 4)
        return fail(SARATHI_ERR_CAPACITY, "host_buf too small (info->packed_ints holds the size needed)");

    int32_t* b = host_buf;
    // every int is written below but the padding before the items
    std::memset(b + info->off_req_aux + ns, 0, (size_t)(info->off_items - info->off_req_aux - ns) * 4);
    int32_t* qo = b + info->off_qo_indptr;
    int32_t* kvp = b + info->off_kv_page_indptr;
    int32_t* kvi = b + info->off_kv_page_indices;
    qo[0] = 0;
    kvp[0] = 0;
    for (int32_t s = 0; s < ns; ++s) {
        const sarathi_request& r = reqs[sched[s].req];
        const int32_t n = sched[s].n;
        b[info->off_req_index + s] = sched[s].req;
        b[info->off_num_new + s] = n;
        b[info->off_last_chunk + s] = (r.state == SARATHI_DECODE || r.num_computed + n == r.prompt_len) ? 1 : 0;
        qo[s + 1] = qo[s] + n;
        std::memcpy(kvi + kvp[s], r.pages, (size_t)np[s] * 4);
        kvp[s + 1] = kvp[s] + np[s];
        b[info->off_kv_last_page_len + s] = r.num_computed + n - kPage * (np[s] - 1);
        b[info->off_req_aux + s] = aux[s];
    }
    int32_t* items = b + info->off_items;
    int64_t w = 0;
    auto put = [&](const ItemHead& src, int32_t b0 = 0, int32_t b1 = 0, int32_t piece = 0) {
        int32_t* it = items + kItemInts * w++;
        std::memcpy(it, src.data(), sizeof src);
        const int32_t s = it[kS];
        it[kQo0] = qo[s];
        it[kNNew] = qo[s + 1] - qo[s];
        it[kKvp0] = kvp[s];
        it[kNp] = np[s];
        it[kKvLen] = kPage * (np[s] - 1) + b[info->off_kv_last_page_len + s];
        for (int k = kKvLen + 1; k < kIds; ++k) it[k] = 0;
        it[kB0] = b0;
        it[kB1] = b1;
        it[kPiece] = piece;
        int32_t* ids = it + kIds;
        if (it[kKind] == kDecode) {
            for (int k = 0; k < kItemIds; ++k) ids[k] = k < it[kCount] ? kvi[kvp[s] + it[kStart] + k] : 0;
        } else if (it[kKind] == kPrefill) {
            const int32_t p0 = b0 * (kTileRows / kPage);  // the pages of the item's first block
            for (int k = 0; k < kItemIds; ++k) ids[k] = p0 + k < np[s] ? kvi[kvp[s] + p0 + k] : 0;
        } else {
            for (int k = 0; k < kItemIds; ++k) ids[k] = 0;
        }
    };
    // the first queue, then the second
    if (apps_first)
        for (auto& a : appends) put(a);
    for (size_t i = 0; i < n_tiles - (size_t)split_k; ++i) put(tiles[pf_order[i]].it);
    int32_t mg = piece_merge0;
    for (size_t i = n_tiles - (size_t)split_k; i < n_tiles; ++i) {
        const ItemHead& t = tiles[pf_order[i]].it;
        const int32_t nb = tile_blocks(t);
        if (nb < 2 * split_n) {
            put(t);
            continue;
        }
        ItemHead h = t;
        h[kSlot] = piece_slot0;
        h[kMerge] = mg++;
        h[kNSplit] = split_n;
        for (int32_t k = 0; k < split_n; ++k) put(h, (int32_t)((int64_t)nb * k / split_n), (int32_t)((int64_t)nb * (k + 1) / split_n), k);
        piece_slot0 += split_n * pf_piece_slots(group);
    }
    if (!apps_first)
        for (auto& a : appends) put(a);
    for (uint32_t i : dec_order) put(decs[i].it);
    set_error("");
    return (policy->kind == SARATHI_POLICY_STALL_FREE && decodes > token_budget) ? SARATHI_WARN_OVER_BUDGET_DECODES
                                                                                 : SARATHI_OK;
}

extern "C" int32_t sarathi_advance(sarathi_request* reqs, int32_t n_reqs, const sarathi_plan_info* info,
                                   const int32_t* host_buf) {
    if (!info || !host_buf || (n_reqs > 0 && !reqs)) return fail(SARATHI_ERR_INVALID_ARG, "NULL pointer");
    const int32_t* req_index = host_buf + info->off_req_index;
    const int32_t* num_new = host_buf + info->off_num_new;
    for (int32_t s = 0; s < info->n_sched; ++s) {
        const int32_t i = req_index[s], n = num_new[s];
        if (i < 0 || i >= n_reqs || n <= 0) return fail(SARATHI_ERR_INVALID_ARG, "plan row out of range");
        sarathi_request& r = reqs[i];
        r.num_computed += n;
        if (r.state == SARATHI_DECODE) continue;
        if (r.num_computed > r.prompt_len) return fail(SARATHI_ERR_INVALID_ARG, "chunk past the prompt");
        r.state = r.num_computed == r.prompt_len ? SARATHI_DECODE : SARATHI_PREFILL_RUNNING;
    }
    set_error("");
    return SARATHI_OK;
}

extern "C" int32_t sarathi_split_metadata(const sarathi_plan_info* info, const int32_t* host_buf, int32_t* out,
                                          size_t out_bytes, sarathi_meta_set* decode, sarathi_meta_set* prefill) {
    if (!info || !host_buf || !out || !decode || !prefill) return fail(SARATHI_ERR_INVALID_ARG, "NULL pointer");
    const int64_t need = 3 * (int64_t)info->n_sched + 4 + info->nnz_pages;
    if ((int64_t)(out_bytes / 4) < need) return fail(SARATHI_ERR_CAPACITY, "split buffer too small");
    const int32_t* qo = host_buf + info->off_qo_indptr;
    const int32_t* kvp = host_buf + info->off_kv_page_indptr;
    const int32_t* kvi = host_buf + info->off_kv_page_indices;
    const int32_t* last = host_buf + info->off_kv_last_page_len;
    int64_t off = 0;
    auto emit = [&](sarathi_meta_set* m, int32_t r0, int32_t r1) {
        m->rows = r1 - r0;
        m->first_row = r0;
        m->token_offset = qo[r0];
        m->tokens = qo[r1] - qo[r0];
        m->nnz_pages = kvp[r1] - kvp[r0];
        m->off_qo_indptr = (int32_t)off;
        for (int32_t s = r0; s <= r1; ++s) out[off++] = qo[s] - qo[r0];
        m->off_kv_page_indptr = (int32_t)off;
        for (int32_t s = r0; s <= r1; ++s) out[off++] = kvp[s] - kvp[r0];
        m->off_kv_page_indices = (int32_t)off;
        for (int32_t p = kvp[r0]; p < kvp[r1]; ++p) out[off++] = kvi[p];
        m->off_kv_last_page_len = (int32_t)off;
        for (int32_t s = r0; s < r1; ++s) out[off++] = last[s];
    };
    emit(decode, 0, info->num_decodes);
    emit(prefill, info->num_decodes, info->n_sched);
    set_error("");
    return SARATHI_OK;
}

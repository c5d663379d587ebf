// sarathi_internal.h -- layout contract between the host planner (plan.cpp)
// and the step kernel (mixed_attn.cu).  Not part of the public ABI.
#pragma once
#include <stdint.h>

struct sarathi_shape;

namespace sarathi {

// Error helpers shared by the planner and the launcher (thread-local message).
void set_error(const char* msg);
int32_t fail(int32_t code, const char* msg);
int32_t check_shape(const sarathi_shape* shape);

constexpr int kPage = 16;             // tokens per KV page (the only size built)
constexpr int kAppendHeads = 2;       // kv heads per APPEND work item (its tokens: one 128-position block's)
constexpr int kAppendBufs = 8;        // mbarriers of an APPEND item (one per page)
constexpr int kTileRows = 128;        // query rows (token x head-in-group) per prefill tile
constexpr int kMaxGroup = 16;         // q heads per kv head handled by the decode path
constexpr int kDecodeMinSplitPages = 8;
constexpr int kDecodeItemsPerSm = 2;  // target split-KV items per SM for the decode phase
constexpr int kDecodeHeads = 2;       // kv heads per decode item (4 streaming warps each)
constexpr int kItemInts = 24;
constexpr int kItemIds = 8;           // page ids carried in an item (one per decode warp)

enum ItemKind : int32_t { kAppend = 0, kPrefill = 1, kDecode = 2 };

// Work item, kItemInts int32 (96 bytes, 16-byte aligned):
//   [0] kind
//   [1] s        scheduled row (request) index
//   [2] g        kv head (prefill); first of the item's kv heads (append: up to
//                kAppendHeads, decode: up to kDecodeHeads)
//   [3] start    append: first token (request-local); prefill: first token of the
//                item's Q tile (request-local); decode: first page (request-local)
//   [4] count    tokens (append / prefill) or pages (decode)
//   [5] slot     decode: first partial slot of its merge group (the group's
//                splits own consecutive slots; split k = start / ceil(pages /
//                nsplit) owns slots slot + k h .. + h - 1 for its h kv heads,
//                one per head); prefill key piece: the tile's first
//                slot (piece k owns pf_piece_slots slots from slot + k times
//                that); -1 when the item is the only split
//   [6] merge    decode / key piece: merge group, -1 when the item is the only split
//   [7] nsplit   decode / key piece: splits in the merge group
//   [8..12]      row s: qo_indptr[s], new tokens, kv_page_indptr[s], pages,
//                kv length -- copies of the metadata, so that an item needs
//                one load before its first page can be fetched
//   [13..15]     prefill: the item's 128-key blocks [b0, b1) and its piece
//                index when its tile is split along the keys (then [5..7] are
//                the tile's first partial slot, merge group and piece count,
//                as for decode splits); 0, 0, 0: the whole tile
//   [16..23]     decode: the page id of page start + w for decode warp w (0
//                past the item's pages); prefill: the ids of the pages of its
//                first block (0 past the request's pages); append: zero
enum ItemField { kKind = 0, kS, kG, kStart, kCount, kSlot, kMerge, kNSplit, kQo0, kNNew, kKvp0, kNp, kKvLen,
                 kB0, kB1, kPiece, kIds = 16 };

// Workspace: an int32 header, then fp32 partial slots from a 256-byte boundary.
//   [0] second queue's head   [1] CTAs exited   [2] error word   [3] error detail
//   [4..11] where a bounded wait ran out   [12] first queue's head
//   [kHdrInts + f]             ready flags of the chunks' K/V: one word per
//                              (row, 128-position block holding some of the
//                              row's new tokens, group of kAppendHeads kv
//                              heads), set to 1 by the APPEND item that wrote
//                              it; row s's flags start at its req_aux entry
//   [kHdrInts + F + m]         arrivals in merge group m (F = flag_ints)
constexpr int kHdrInts = 16;
constexpr int kErrWait = 1;     // a bounded wait ran out
constexpr int kErrBounds = 2;   // a bounds check failed

#if defined(__CUDACC__)
#define SARATHI_HD __host__ __device__
#else
#define SARATHI_HD
#endif
SARATHI_HD inline int kv_groups(int Hkv) { return (Hkv + kAppendHeads - 1) / kAppendHeads; }
// A row of n new tokens touches at most n / 128 + 2 blocks of 128 positions.
inline int64_t flag_ints(int n_sched, int num_tokens, int Hkv) {
    return ((int64_t)num_tokens / kTileRows + 2 * (int64_t)n_sched) * kv_groups(Hkv);
}
inline int64_t sync_ints(int n_sched, int n_merge, int num_tokens, int Hkv) {
    return kHdrInts + flag_ints(n_sched, num_tokens, Hkv) + n_merge;
}
inline int64_t partial_offset_bytes(int n_sched, int n_merge, int num_tokens, int Hkv) {
    int64_t b = sync_ints(n_sched, n_merge, num_tokens, Hkv) * 4;
    return (b + 255) / 256 * 256;
}
// One decode split writes, for each q head of its group, o[d] (normalised by
// its own sum), then m and l (running max and sum, base-2 logits).
inline int64_t partial_slot_floats(int group, int d) { return (int64_t)group * (d + 2); }

inline int tokens_per_tile(int group) { return group >= kTileRows ? 1 : kTileRows / group; }
// A prefill tile split along its keys runs as 2..kMaxPieces pieces; each
// piece's partial ([128][d] fp32 O / l, then m[128], l[128]) takes
// pf_piece_slots(group) partial slots: an even count when the group is odd,
// so that every piece's partial starts on a 16-byte boundary (the first slot
// of a split tile is even too).
constexpr int kMaxPieces = 4;
SARATHI_HD inline int pf_piece_slots(int group) {
    const int n = (kTileRows + group - 1) / group;
    return (group & 1) ? (n + 1) / 2 * 2 : n;
}
// A prefill item is one Q tile.
inline int tokens_per_item(int group) { return tokens_per_tile(group); }

}  // namespace sarathi

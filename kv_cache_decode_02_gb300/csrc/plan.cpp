// Compact indirect cell plan, built on the host ("KVARN KV Performance optimizations",
// item 3: a capacity-sized duplicate bitmap with first-occurrence semantics, capacity
// checks and sentinel padding; item 4: cells grouped by their physical 128-cell record,
// records sorted by physical id, one complete monotonic segment per selected record with
// -1 holes kept; item 5: the physical cell is the low 32 bits of the encoded index, the
// high bits carry stage-slot metadata that a read plan does not need).
//
// A segment is positional -- entry j of record r's segment is r*128 + j or -1 -- so a
// split aligned to 128 entries reads exactly one contiguous physical record.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "kvattn_internal.cuh"

namespace kvattn {

namespace {
constexpr int64_t kRecord = 128;
}

int build_cell_plan_host(const int64_t* cells, const int64_t* offsets, int n_seq,
                         int64_t capacity_cells, int32_t* plan, int64_t plan_stride,
                         int32_t* seq_lens) {
    if (n_seq < 0 || capacity_cells < 1 || capacity_cells > (int64_t)INT32_MAX + 1 ||
        plan_stride < 0)
        return KVATTN_ERR_INVALID_ARG;
    if (n_seq == 0) return KVATTN_OK;
    if (offsets == nullptr || seq_lens == nullptr) return KVATTN_ERR_INVALID_ARG;
    if (offsets[0] != 0) return KVATTN_ERR_INVALID_ARG;
    for (int s = 0; s < n_seq; ++s)
        if (offsets[s + 1] < offsets[s]) return KVATTN_ERR_INVALID_ARG;
    if (offsets[n_seq] > 0 && cells == nullptr) return KVATTN_ERR_INVALID_ARG;

    const int64_t n_records = (capacity_cells + kRecord - 1) / kRecord;
    std::vector<uint64_t> cell_bits;     // one bit per physical cell, 2 words per record
    std::vector<uint8_t> record_seen;    // one flag per record
    std::vector<int64_t> records;
    try {
        cell_bits.assign((size_t)n_records * 2, 0);
        record_seen.assign((size_t)n_records, 0);
    } catch (const std::bad_alloc&) {
        return KVATTN_ERR_INVALID_ARG;
    }

    for (int s = 0; s < n_seq; ++s) {
        records.clear();
        int status = KVATTN_OK;
        for (int64_t k = offsets[s]; k < offsets[s + 1]; ++k) {
            const uint64_t c = (uint64_t)cells[k] & 0xffffffffull;  // low 32 bits, unsigned
            if ((int64_t)c >= capacity_cells) {
                status = KVATTN_ERR_CAPACITY;
                break;
            }
            uint64_t& word = cell_bits[c >> 6];
            const uint64_t bit = 1ull << (c & 63);
            if (word & bit) continue;  // a later duplicate: the first occurrence already counts
            word |= bit;
            const int64_t r = (int64_t)(c / kRecord);
            if (!record_seen[r]) {
                record_seen[r] = 1;
                records.push_back(r);
            }
        }
        std::sort(records.begin(), records.end());
        const int64_t len = (int64_t)records.size() * kRecord;
        if (status == KVATTN_OK && len > INT32_MAX) status = KVATTN_ERR_CAPACITY;
        if (status == KVATTN_OK && plan != nullptr && len > plan_stride) status = KVATTN_ERR_CAPACITY;
        if (status == KVATTN_OK) {
            seq_lens[s] = (int32_t)len;
            if (plan != nullptr) {
                int32_t* row = plan + (int64_t)s * plan_stride;
                int64_t pos = 0;
                for (int64_t r : records) {
                    const uint64_t w0 = cell_bits[2 * r], w1 = cell_bits[2 * r + 1];
                    for (int64_t j = 0; j < kRecord; ++j) {
                        const uint64_t w = j < 64 ? w0 : w1;
                        const bool sel = (w >> (j & 63)) & 1ull;
                        row[pos++] = sel ? (int32_t)(r * kRecord + j) : -1;
                    }
                }
                for (; pos < plan_stride; ++pos) row[pos] = -1;
            }
        }
        // reset only what this sequence touched (every touched record was pushed)
        for (int64_t r : records) {
            cell_bits[2 * r] = cell_bits[2 * r + 1] = 0;
            record_seen[r] = 0;
        }
        if (status != KVATTN_OK) return status;
    }
    return KVATTN_OK;
}

}  // namespace kvattn

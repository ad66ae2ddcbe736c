// Host-side ranks builder: token histogram, frequency-ranked shortlist after
// a forced id set, and the sorted union of two id lists.  No GPU involved.
// ("Shortlist MTP", section "Building the 16k shortlist": every id below
// 8,192, a structural core, then the most frequent remaining ids until the
// list is full; "[DGX Spark] Qwen3.8-Flash-Next on two DGX Sparks", section
// "Build the draft vocabulary from your own text": count a corpus's tokens,
// write an id list of a given size, merge it with an existing list as a
// sorted set union.)
#include <algorithm>
#include <cstdint>
#include <vector>

#include "dvl.h"

namespace {

// Rank order: more frequent first; equal counts by ascending id.
struct RankLess {
    const int64_t *c;
    bool operator()(int32_t a, int32_t b) const { return c[a] != c[b] ? c[a] > c[b] : a < b; }
};

}  // namespace

extern "C" {

dvl_status dvl_histogram(const int32_t *tokens, int64_t n, int64_t V, int64_t *counts)
{
    if (n < 0 || V < 1 || !counts || (n > 0 && !tokens))
        return DVL_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (tokens[i] < 0 || (int64_t)tokens[i] >= V)
            return DVL_ERR_OUT_OF_RANGE;
    for (int64_t i = 0; i < n; ++i)
        ++counts[tokens[i]];
    return DVL_OK;
}

dvl_status dvl_build_ranks(const int64_t *counts, int64_t V, const int32_t *forced,
                           int32_t n_forced, int32_t N, int32_t sorted, int32_t *ranks_out,
                           int32_t *n_out)
{
    if (!counts || V < 1 || V > 0x7fffffffLL || N < 0 || n_forced < 0 || !n_out ||
        (n_forced > 0 && !forced) || (N > 0 && !ranks_out))
        return DVL_ERR_INVALID_ARG;
    std::vector<unsigned char> in_forced((size_t)V, 0);
    std::vector<int32_t> head;
    head.reserve((size_t)n_forced);
    for (int32_t i = 0; i < n_forced; ++i) {
        const int32_t f = forced[i];
        if (f < 0 || (int64_t)f >= V)
            return DVL_ERR_OUT_OF_RANGE;
        if (!in_forced[(size_t)f]) {
            in_forced[(size_t)f] = 1;
            head.push_back(f);
        }
    }
    const RankLess less{counts};
    std::sort(head.begin(), head.end(), less);
    const int64_t total = std::min<int64_t>(N, V);
    const int64_t want_rest = std::max<int64_t>(0, total - (int64_t)head.size());
    std::vector<int32_t> rest;
    rest.reserve((size_t)(V - (int64_t)head.size()));
    for (int64_t t = 0; t < V; ++t)
        if (!in_forced[(size_t)t])
            rest.push_back((int32_t)t);
    const int64_t take = std::min<int64_t>(want_rest, (int64_t)rest.size());
    std::partial_sort(rest.begin(), rest.begin() + take, rest.end(), less);
    int64_t w = 0;
    for (size_t i = 0; i < head.size() && w < total; ++i)
        ranks_out[w++] = head[i];
    for (int64_t i = 0; i < take && w < total; ++i)
        ranks_out[w++] = rest[(size_t)i];
    if (sorted)
        std::sort(ranks_out, ranks_out + w);
    *n_out = (int32_t)w;
    return DVL_OK;
}

dvl_status dvl_union_sorted(const int32_t *a, int32_t na, const int32_t *b, int32_t nb,
                            int32_t *out, int32_t *n_out)
{
    if (na < 0 || nb < 0 || !n_out || (na > 0 && !a) || (nb > 0 && !b) ||
        (na + nb > 0 && !out))
        return DVL_ERR_INVALID_ARG;
    std::vector<int32_t> sa(a, a + na), sb(b, b + nb);
    std::sort(sa.begin(), sa.end());
    sa.erase(std::unique(sa.begin(), sa.end()), sa.end());
    std::sort(sb.begin(), sb.end());
    sb.erase(std::unique(sb.begin(), sb.end()), sb.end());
    int32_t *end = std::set_union(sa.begin(), sa.end(), sb.begin(), sb.end(), out);
    *n_out = (int32_t)(end - out);
    return DVL_OK;
}

}  // extern "C"

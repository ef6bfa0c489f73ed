// Measured dispatch table: for a (N, K) pair and an M range, the variant and
// launch parameters that ran fastest in the tuning sweep.  Entries come from
// tuning_table.inc, which the sweep script writes; shapes it does not list
// fall back to the dispatcher's rules.
#pragma once

#include <stdint.h>

namespace w8a8 {

struct TableEntry {
    int64_t m_lo, m_hi, n, k;
    int variant, split_k, m_tile, block_n_tile, stages;
};

static const TableEntry kTunedTable[] = {
#include "tuning_table.inc"
    {0, 0, 0, 0, 0, 0, 0, 0, 0},
};

inline const TableEntry *lookup_tuned(int64_t M, int64_t N, int64_t K)
{
    for (const TableEntry &e : kTunedTable)
        if (e.n == N && e.k == K && M >= e.m_lo && M <= e.m_hi)
            return &e;
    return nullptr;
}

}  // namespace w8a8

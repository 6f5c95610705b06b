// dg_rows.h -- the one list of decode row buckets.  The table parser, the
// selector, the sweep and the Python binding all derive their rows from here
// (Strata PR #1297, "The second commit: the seam rework", item 3: one rows list).
#pragma once

#define DG_ROWS_BUCKETS(X) X(1) X(2) X(3) X(4) X(6) X(8) X(12) X(16) X(24) X(32) X(48) X(64) X(96) X(128) \
    X(192) X(256) X(384) X(512)
#define DG_ROWS_AS_LIST(m) m,

namespace dg {
int bucket_rows(int M);          // smallest bucket >= M, or -1 when M > 512
const char* op_key_name(int op); // table name of an op
}  // namespace dg

// Host build of the kernels' visible-range and split-partition helpers
// (pa::visible_range, pa::split_bounds, compiled for the host from the same
// header the kernels include), so a CPU test can set them beside the oracle's
// partition.  Test infrastructure only: nothing in the library uses it.
#include "pa_internal.h"

extern "C" void probe_split_bounds(int pos, int seq_len, int causal, int window, int splits, int s, int ps,
                                   long long *lo, long long *hi, long long *j0, long long *j1) {
    int64_t l, h, a, b;
    pa::visible_range(pos, seq_len, causal, window, l, h);
    pa::split_bounds(l, h, splits, s, ps, a, b);
    *lo = l;
    *hi = h;
    *j0 = a;
    *j1 = b;
}

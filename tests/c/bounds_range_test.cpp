// Host test of the range predicate of the checked build (bounds_range.h):
// buffers at the bottom and top of the address space, empty and full-size
// accesses, and sizes whose sum with the address would wrap.
#include <cstdint>
#include <cstdio>

#include "bounds_range.h"

static int failures = 0;

static void expect(bool got, bool want, const char *what)
{
    if (got != want) {
        std::printf("FAIL %s: got %d want %d\n", what, int(got), int(want));
        ++failures;
    }
}

int main()
{
    using dsv4::range_inside;
    const uintptr_t base = 0x1000;
    expect(range_inside(base, 16, base, 64), true, "first bytes");
    expect(range_inside(base + 48, 16, base, 64), true, "last bytes");
    expect(range_inside(base + 49, 16, base, 64), false, "one byte past the end");
    expect(range_inside(base + 64, 0, base, 64), true, "empty access at the end");
    expect(range_inside(base + 64, 1, base, 64), false, "one byte at the end");
    expect(range_inside(base - 1, 1, base, 64), false, "one byte before the start");
    expect(range_inside(base - 16, 32, base, 64), false, "straddles the start");
    expect(range_inside(base, 65, base, 64), false, "longer than the buffer");
    expect(range_inside(base, 64, base, 64), true, "the whole buffer");
    // sizes that would wrap an address sum
    expect(range_inside(base + 8, UINT64_MAX, base, 64), false, "huge size");
    expect(range_inside(UINTPTR_MAX - 7, 8, UINTPTR_MAX - 63, 64), true, "top of the address space");
    expect(range_inside(UINTPTR_MAX - 7, 16, UINTPTR_MAX - 63, 64), false, "past the top");
    expect(range_inside(base + (uint64_t(1) << 40), 16, base, uint64_t(1) << 41), true,
           "offset past 2^32");
    expect(range_inside(base + (uint64_t(1) << 41), 16, base, uint64_t(1) << 41), false,
           "at the end of a 2 TiB buffer");
    std::printf(failures ? "FAILED\n" : "OK\n");
    return failures ? 1 : 0;
}

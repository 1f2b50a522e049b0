"""The fine kernel's epilogue staging layout, checked by enumeration.

Each softmax warp stages its 16 query columns x 32 channels of O (fp32) in 2 KB
of shared memory, word (column c, channel d) at 32 c + ((d + 4 (c & 1)) mod 32).
It writes one column at a time (lane = channel) and reads back 16 bytes a lane:
lane l takes column c = (l >> 2) + 8 j and channels 8 (l & 3) .. + 7 as two
float4 loads. Shared memory has 32 four-byte banks; a 16-byte access is served
eight lanes at a time. This test checks that the layout is a bijection, and that
neither the writes nor the reads conflict.
"""

COLS, CH, BANKS = 16, 32, 32


def word(c, d):
    return 32 * c + ((d + 4 * (c & 1)) % 32)


def test_layout_is_a_bijection_onto_the_warps_2kb():
    words = {word(c, d) for c in range(COLS) for d in range(CH)}
    assert words == set(range(COLS * CH))


def test_column_writes_hit_32_distinct_banks():
    for c in range(COLS):
        banks = {word(c, lane) % BANKS for lane in range(32)}
        assert len(banks) == 32, c


def test_16_byte_reads_are_conflict_free_and_contiguous():
    for j in range(2):
        for half in range(2):  # the two float4 loads: channels 8k .. 8k+3, then 8k+4 .. 8k+7
            for phase in range(4):  # lanes 8 phase .. 8 phase + 7 are served together
                groups = set()
                for lane in range(8 * phase, 8 * phase + 8):
                    c = (lane >> 2) + 8 * j
                    d0 = 8 * (lane & 3) + 4 * half
                    w = [word(c, d0 + e) for e in range(4)]
                    # the kernel reads one float4 at the first word: the four channels sit in
                    # consecutive words, 16-byte aligned
                    assert w == list(range(w[0], w[0] + 4)) and w[0] % 4 == 0, (lane, j, half)
                    groups.add((w[0] % BANKS) // 4)
                assert len(groups) == 8, (j, half, phase)

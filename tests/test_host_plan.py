"""Host-side plan logic, on the CPU: the shape table's choices and the
stream-K schedule (sgemm_table_choice, sgemm_streamk_schedule -- pure host
arithmetic, no CUDA call).

The schedule test carries a model of the kernel's side of the stream-K
protocol (which CTA publishes a partial tile for which tile, and whom each
finisher waits for), so a schedule that would leave a finisher waiting on a
CTA that never publishes fails here instead of timing out on a GPU."""
import itertools

import pytest

import dense_fp32_matrix_sm_gb300 as sg

SMS = 152  # GB300


@pytest.mark.parametrize("case", [
    # (M, N, K, lda, ldb, batch, b_trans) -> (variant, repack A, repack B)
    ((4096, 4096, 4096, None, None, 1, False), ("tmat_128x256x32_s3_b1", False, False)),
    ((4092, 4092, 4092, None, None, 1, False), ("tmat_128x256x32_s3_b1", False, False)),
    ((8192, 14336, 4096, None, None, 1, False), ("tmat_128x256x32_s3_b1", False, False)),
    ((4096, 4096, 4096, 4097, None, 1, False), ("tmat_128x256x32_s3_b1", True, False)),   # padded copy of A
    ((4096, 4096, 4096, None, 4097, 1, False), ("tmat_128x256x32_s3_b1", False, True)),   # ... of B
    ((1, 16384, 8192, None, None, 1, False), ("gemv_4x512", False, False)),
    ((4, 16384, 8192, None, None, 1, True), ("gemv_4x512", False, False)),                # B given transposed
    ((16, 16384, 8192, None, None, 1, False), ("gemv_16x1024", False, False)),
    ((16, 16384, 8192, None, None, 1, True), ("skinny_sk_16x128x32_w4_s3_b3_ef", False, False)),
    ((128, 128, 128, None, None, 1, False), ("tiny_32x32", False, False)),
    ((512, 512, 512, None, None, 1, False), ("tiny_32x32", False, False)),
    ((200, 130, 100, 101, 131, 1, False), ("tiny_32x32", False, False)),                 # any layout, no copy
    ((32, 4096, 4096, None, None, 1, False), ("tiny_32x32", False, False)),              # 17-32 rows, long K
    ((20, 3000, 2000, None, None, 1, False), ("tmat_64x256x32_s3_b1", False, False)),    # too few 32x32 tiles
    ((64, 16384, 8192, None, None, 1, False), ("tmat_64x256x32_s3_b1", False, False)),
    ((48, 2048, 1024, None, None, 3, False), ("tmat_64x256x32_s3_b1", False, False)),    # a strided batch
    ((768, 768, 512, None, None, 1, False), ("small_64x64", False, False)),
    ((1024, 1024, 256, None, None, 1, False), ("small_64x64", False, False)),
    ((1024, 1024, 512, None, None, 1, False), ("tmat_128x128x32_s4_b1", False, False)),  # 256 tiles: unbalanced
    ((1408, 1408, 1408, None, None, 1, False), ("tmat_128x128x32_s4_b1", False, False)), # last 256-col tile half empty
    ((1280, 1280, 1280, None, None, 1, False), ("tmat_128x256x32_s3_b1", False, False)),
    ((1536, 1536, 256, None, None, 1, False), ("tmat_128x128x32_s4_b1", False, False)),  # short K, < 3/4 wave
    ((2048, 2048, 256, None, None, 1, False), ("tmat_128x256x32_s3_b1", False, False)),
    ((100, 96, 1000, 1001, None, 1, False), ("cpa_128x128x32_s3_k8_b2", False, False)),  # small, odd lda: no copy
    ((100, 96, 1000, None, 97, 1, False), ("generic_64x64x16", False, False)),           # small, odd ldb
])
def test_table_choice(case):
    (M, N, K, lda, ldb, batch, tb), expect = case
    got = sg.table_choice(M, N, K, lda=lda, ldb=ldb, batch=batch, stride_a=M * (lda or K),
                          stride_b=K * (ldb or N), b_trans=tb, num_sms=SMS)
    assert got == expect, (case, got)


def test_table_choice_rejects_bad_arguments():
    for args in [dict(M=-1, N=4, K=4), dict(M=4, N=4, K=4, lda=3), dict(M=4, N=4, K=4, num_sms=0)]:
        with pytest.raises(sg.SgemmError) as e:
            sg.table_choice(**args)
        assert e.value.status == sg.SGEMM_ERR_INVALID_ARG


def kernel_protocol(tiles, KT, grid, dp_waves, sk_iters):
    """The kernel's view of a schedule: CTA b takes data-parallel tiles
    b + i*grid (i < dp_waves) and the k-slices [b*I/grid, (b+1)*I/grid) of the
    tail tiles (tile-major, I = sk_iters), cut at tile boundaries into at most
    two segments.  A segment that ends before its tile's last slice publishes
    a partial tile; the one that holds the last slice (and not the first)
    waits for every CTA from the first one holding a slice of the tile up to
    itself.  Returns (publishers per tile, waited-on CTAs per tile, slices
    covered per tile)."""
    publish, waits, covered = {}, {}, {}
    t0 = dp_waves * grid
    for b in range(grid):
        for i in range(dp_waves):
            covered[b + i * grid] = covered.get(b + i * grid, 0) + KT
        if sk_iters == 0:
            continue
        s0, e0 = b * sk_iters // grid, (b + 1) * sk_iters // grid
        if s0 >= e0:
            continue
        tf, tl = s0 // KT, (e0 - 1) // KT
        assert tl - tf <= 1, "a range spans more than two tiles"
        segs = [(tl, 0, e0 - tl * KT), (tf, s0 - tf * KT, KT)] if tl != tf else \
            [(tf, s0 - tf * KT, e0 - tf * KT)]
        for (t, k0, k1) in segs:
            covered[t0 + t] = covered.get(t0 + t, 0) + (k1 - k0)
            if k1 < KT:
                publish.setdefault(t, set()).add(b)
            elif k0 > 0:
                c_first = ((t * KT + 1) * grid - 1) // sk_iters
                waits[t] = set(range(c_first, b))
    return publish, waits, covered


@pytest.mark.parametrize("ctas_per_sm", [1, 2])
def test_streamk_schedule_keeps_every_wait_satisfiable(ctas_per_sm):
    slots = SMS * ctas_per_sm
    checked = 0
    for tiles, KT in itertools.product(list(range(1, 40)) + list(range(140, 170)) + [300, 303, 304, 305, 456, 457,
                                                                                      512, 3584],
                                       [1, 2, 7, 8, 9, 16, 32, 33, 128]):
        grid, dp, I = sg.streamk_schedule(tiles, KT, SMS, ctas_per_sm)
        assert 1 <= grid <= max(slots, tiles)
        if I == 0:
            # no split: a plain persistent grid over whole tiles
            assert dp == 0 and grid == min(tiles, slots)
            continue
        checked += 1
        assert I >= grid, (tiles, KT, grid, I)          # every CTA holds at least one slice
        assert I % KT == 0 and dp * grid + I // KT == tiles
        publish, waits, covered = kernel_protocol(tiles, KT, grid, dp, I)
        assert all(covered.get(t, 0) == KT for t in range(tiles)), (tiles, KT)
        for t, pub in publish.items():
            assert waits.get(t) == pub, (tiles, KT, grid, t)
        assert set(waits) <= set(publish)
    assert checked > 50


def test_streamk_schedule_examples():
    # 4096^3 on 128 x 256 tiles: 3 waves, then 56 tiles x 128 slices shared by 152 CTAs
    assert sg.streamk_schedule(512, 128) == (152, 3, 56 * 128)
    # fewer tiles than CTAs: every tile split, no data-parallel wave
    assert sg.streamk_schedule(81, 8) == (152, 0, 648)
    # a tail of 10 tiles x 8 slices for 152 CTAs would leave CTAs without a slice: a plain partial wave
    assert sg.streamk_schedule(162, 8) == (152, 0, 0)
    with pytest.raises(sg.SgemmError):
        sg.streamk_schedule(-1, 8)

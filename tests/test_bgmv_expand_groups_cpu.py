"""CPU restatement of the BGMV expand's work split when a unit's token tiles run
side by side on thread groups (column chunks narrower than half the block's
reach): for every chunk width, unit length and group count the kernel can take,
each (token, column) of the unit is produced by exactly one thread exactly once,
the u rows a group reads stay inside the pass's staged rows, and the rows window
of 32 tokens is reloaded only at multiples of a pass."""
import pytest

THREADS, TT, REACH, ROWS_WIN = 256, 4, 256 * 4, 32


def _group_count(pw, cnt):
    """The kernel's choice: groups only where pw * 2 <= reach; then up to four, never more than the tiles."""
    if pw * 2 > REACH:
        return 1
    ng_geo = 4 if pw * 4 <= REACH else 2
    ntiles = (cnt + TT - 1) // TT
    return min(ng_geo, 4 if ntiles >= 3 else ntiles)


@pytest.mark.parametrize("pw", [64, 128, 256, 512, 1024, 2048])
def test_every_output_once(pw):
    for pcn in sorted({pw, pw - 8, 8, max(8, pw // 2 + 8)}):
        if pcn > pw or pcn <= 0:
            continue
        for cnt in list(range(1, 41)) + [63, 64, 65, 130]:
            ng = _group_count(pw, cnt)
            gs, tpp = THREADS // ng, TT * ng
            npass = (cnt + tpp - 1) // tpp
            assert ROWS_WIN % tpp == 0                     # windows start at pass boundaries
            seen = {}
            for p in range(npass):
                for tid in range(THREADS):
                    grp, lt = tid // gs, tid % gs
                    tok0 = p * tpp + grp * TT
                    nt = min(TT, cnt - tok0)
                    if nt <= 0:
                        continue
                    u_row0 = grp * TT                          # rows of the pass's staged u this group reads
                    assert 0 <= u_row0 and u_row0 + TT <= tpp
                    for cq in range(lt * 4, pcn, gs * 4):
                        for t in range(nt):
                            for c in range(cq, min(cq + 4, pcn)):
                                key = (tok0 + t, c)
                                seen[key] = seen.get(key, 0) + 1
            assert len(seen) == cnt * pcn, (pw, pcn, cnt, ng)
            assert set(seen.values()) == {1}, (pw, pcn, cnt, ng)

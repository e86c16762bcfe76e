"""Apply allocator operations to the oracle model or the library's allocator
with one interface: each call returns a result or the string "capacity" /
"arg" for a typed error."""
from oracle import allocator as OA


def run_oracle(a, op):
    try:
        return _call(a, op)
    except OA.CapacityError:
        return "capacity"
    except OA.ArgError:
        return "arg"


def run_native(a, op):
    from paged_kv_decode_09_gb300 import api
    try:
        return _call(a, op)
    except api.PkvError as e:
        return {3: "capacity", 1: "arg"}.get(e.status, f"status{e.status}")


def _call(a, op):
    k = op["op"]
    if k == "open":
        return a.open()
    if k == "fork":
        return a.fork(op["seq"])
    if k in ("reserve", "commit", "unreserve"):
        getattr(a, k)(op["seq"], op["n"])
        return None
    if k in ("reserve_many", "commit_many"):
        getattr(a, k)(op["seqs"], op["n"])
        return None
    if k == "release":
        a.release(op["seq"])
        return None
    if k == "info":
        return list(a.info(op["seq"]))
    if k == "block_table":
        return [int(x) for x in a.block_table(op["seq"], op["stride"])]
    if k == "batch":
        rows, lens = a.batch(op["seqs"], op["extra"], op["stride"])
        return [[[int(x) for x in r] for r in rows], [int(x) for x in lens]]
    if k == "stats":
        return list(a.stats())
    if k == "page_refs":
        return a.page_refs(op["page"]) if hasattr(a, "page_refs") else a.refs[op["page"]]
    raise ValueError(k)

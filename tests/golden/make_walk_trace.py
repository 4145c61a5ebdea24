"""Writes walk_trace.json: the slots of the page-3 walk ("Paged KV Cache - AI
infra interview lesson", Walk the Shapes First, block_size 4, 8 blocks).

The page prints sequence A's prefill slots ([28, 29, 30, 31, 8, 9] for its
blocks [7, 2]) and the rules; its table of the later steps did not survive
extraction.  This script derives every step with the oracle only:
  * the allocation (which block a sequence takes when it needs a new one) by
    the oracle's allocator model, oracle/block_allocator.py (lowest-numbered
    free block first: B's fifth token takes block 0);
  * the slots by the oracle's slot mapping, oracle.compute_slot_mapping, over
    the positions each step writes ([start, end) per sequence).

    python tests/golden/make_walk_trace.py          # rewrites the file
    python tests/golden/make_walk_trace.py --check  # exit 1 if it differs
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

BLOCK_SIZE, NUM_BLOCKS, MAX_BLOCKS = 4, 8, 3
SOURCE = ("Paged KV Cache - AI infra interview lesson; Walk the Shapes First (block_size 4, A: 6 tokens in blocks "
          "[7, 2], B: 3 tokens in block [5]; the slot of position p is block_table[p // bs] * bs + p % bs; a new "
          "block is needed exactly when len % bs == 1) and Step 1 (A's prefill slots)")


def derive():
    import oracle
    from oracle.block_allocator import ModelAllocator

    alloc = ModelAllocator(NUM_BLOCKS, BLOCK_SIZE)
    alloc.add_sequence("A", 6, blocks=[7, 2])
    alloc.add_sequence("B", 3, blocks=[5])

    def slots(starts, ends):
        tables = [alloc.block_table(s, MAX_BLOCKS)[0] for s in ("A", "B")]
        out, err = oracle.compute_slot_mapping(tables, starts, ends, BLOCK_SIZE, NUM_BLOCKS)
        assert err == 0
        return out.tolist()

    steps = [{"name": "prefill", "slots": slots([0, 0], [6, 3])}]
    for name in ("decode 1", "decode 2"):
        starts = [alloc.seqs[s]["len"] for s in ("A", "B")]
        for s in ("A", "B"):
            alloc.append(s)  # one new token each; a new block when the length becomes 1 mod block_size
        ends = [alloc.seqs[s]["len"] for s in ("A", "B")]
        steps.append({"name": name, "slots": slots(starts, ends)})
    return {
        "source": SOURCE,
        "printed_on_page": {"A_prefill": [28, 29, 30, 31, 8, 9]},
        "derived_by_the_page_rules": {
            "note": "the page's table did not survive extraction; these follow from its stated rules, with B's new "
                    "block taken as the lowest-numbered free block (0)",
            "generated_by": "tests/golden/make_walk_trace.py (oracle.block_allocator.ModelAllocator for the "
                            "allocation, oracle.compute_slot_mapping for the slots)",
            "steps": steps,
        },
    }


def main(argv):
    path = os.path.join(HERE, "walk_trace.json")
    want = derive()
    if "--check" in argv:
        with open(path) as f:
            return 0 if json.load(f) == want else 1
    with open(path, "w") as f:
        json.dump(want, f, indent=2)
        f.write("\n")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))

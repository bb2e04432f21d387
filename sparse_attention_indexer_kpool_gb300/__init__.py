"""DSA kpool token selection + selected-row NoPE MLA decode for GB300 (sm_103a)."""
